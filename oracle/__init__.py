"""CPU oracle for the fused equivariant message (test infrastructure only).

This package is the plain, slow, double-precision definition of what the GPU
library computes. It exists to check the CUDA path, not to run it: only the
test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import it. The product path (the C-ABI library and its
Python binding) never imports, links or calls anything here, and this package
imports nothing from the product.

Modules
  sh     real orthonormal spherical harmonics l <= 3 from the associated
         Legendre definition (Condon-Shortley phase).
  cg     complex Clebsch-Gordan coefficients by Racah's closed formula, and
         their conversion to the real SH basis.
  layer  the channelwise CG tensor product with per-path channel weights (or
         per-edge radial weights W = R.M) and the sum into receivers.
  backward  the chain rule of that layer: gradients of x, w (or R and M)
         and of the edge vectors through the harmonics.
  graph  the radius graph (ordered pairs closer than the cutoff, CSR by
         receiver), with the cutoff decision taken in float32; open
         boundaries, or a periodic orthorhombic box (every image within
         one box length per direction).

sh, cg and layer take the degree as a parameter (l_max = 3 by default, the
Batmobile layer; l_max = 4..6 for the higher-degree variant the blog lists
as future work); the layer reads it from the feature array's last axis,
(l_max+1)^2 components.

Sources (web pages on the Batmobile kernels and on E2Former-V2):
  * "Batmobile CUDA内核优化：等变图神经网络的10-20倍加速策略" (blog post),
    sections "1. 编译时常量", "2. 寄存器中间计算", "3. 操作融合".
  * E2Former-V2 article (seekfood.cn news 876595), section 2.1 (EAAS,
    Lemma 4.1, Eq. 13).

Every oracle function is pinned by a CPU test to something other than
itself (printed constants, closed forms, library routines, invariants,
brute force); see tests/test_oracle_*.py. Nothing here is "parity
unpinned" except the absolute sign of each odd-parity real CG path, which
is a convention (any per-path sign is absorbed by the path weight); it is
fixed by the stated reading "take Im of the real-basis transform".
"""
