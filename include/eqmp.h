/*
 * eqmp.h - C ABI of libeqmp.so: fused equivariant message passing, l <= 3.
 *
 * One layer of the equivariant-GNN edge message.  For every edge e
 * (sender src_e -> receiver i) it evaluates the 16 real orthonormal
 * spherical harmonics Y_e of the edge vector, takes the channelwise
 * Clebsch-Gordan tensor product with the sender's features over all 34
 * triangle-allowed paths (l1, l2 -> l3, all <= 3) with per-path channel
 * weights, and sums the messages into the receiver:
 *
 *   out[i, c, (l3,m3)] = sum_{e -> i} sum_{p=(l1,l2,l3)} W[e,p,c]
 *                          sum_{m1,m2} C_p[m3,m1,m2] x[src_e, c, (l1,m1)] Y_e[(l2,m2)]
 *
 * Sources: "Batmobile CUDA内核优化：等变图神经网络的10-20倍加速策略" (blog
 * post): section "2. 寄存器中间计算" (SH in registers, Y00 and the l = 1
 * constants), section "1. 编译时常量" (34 compile-time CG entries for
 * L_MAX = 3), section "3. 操作融合" (the fused kernel's arguments: edge
 * vectors [E,3], node features [N,C,16], source indices [E]; one read of
 * each edge vector; the message-passing sum as the third fused step).
 *
 * Conventions shared by every entry point
 *   - Component index k = l*l + l + m, m = -l..l (16 per channel); real
 *     SH with the Condon-Shortley phase (Y00 = 0.28209479, Y_1,-1 = -c y,
 *     Y_10 = c z, Y_11 = -c x, c = 0.48860251).
 *   - Path order for weights: l1 = 0..3, l2 = 0..3,
 *     l3 = |l1-l2|..min(3, l1+l2)  (34 paths; eqmp_path_table lists them).
 *     Real CG tables are unit-normalised CG coefficients in the real basis;
 *     the 11 odd-parity paths (l1+l2+l3 odd) are taken as -i times the
 *     (purely imaginary) transform.
 *   - Graph: CSR by receiver.  row_offsets[N+1] holds ABSOLUTE indices into
 *     the edge arrays (vec, Y, src, R); receiver i owns edges
 *     row_offsets[i] .. row_offsets[i+1]-1.  A receiver range [a, b) of a
 *     larger graph is therefore (row_offsets + a, N = b - a, out + a*C*16).
 *   - Every pointer argument except eqmp_path_table's is DEVICE memory,
 *     allocated and owned by the caller.  The library allocates no device
 *     memory and keeps no state between calls beyond a per-device launch
 *     configuration cache and a device-side watchdog flag.
 *   - out is overwritten, never accumulated; receivers with no edges get 0.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream); the
 *     caller synchronises before reading results.
 *   - Precision: SH, CG and all accumulation in fp32.  x and out may be
 *     stored as bf16 (round-to-nearest-even, once, on the final store).
 *   - Errors: arguments are checked on the host before any launch and
 *     reported as a status; nothing traps on the device.  Preconditions not
 *     checked on the host (offsets non-decreasing with 0 <= off <= E,
 *     0 <= src < N_src, finite vectors) cannot make a kernel fault or hang:
 *     indices are clamped, out-of-range senders read as zero features, and
 *     every device-side wait is bounded (see eqmp_device_error).  With them
 *     violated the outputs are unspecified.  eqmp_validate_graph checks them.
 *   - Zero-length edge vectors give n = 0: Y00 stays, every l >= 1 term is 0.
 */
#ifndef EQMP_H
#define EQMP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so C callers need no CUDA headers. */
typedef struct CUstream_st* eqmp_stream_t;

typedef enum {
  EQMP_OK = 0,
  EQMP_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misalignment, bad enum */
  EQMP_ERR_UNSUPPORTED = 2,   /* valid but not built: C not in {8,16,32,64,128}, K != 8 */
  EQMP_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  EQMP_ERR_DEVICE_TIMEOUT = 4,/* a bounded device-side wait gave up (see eqmp_device_error) */
  EQMP_ERR_GRAPH = 5          /* eqmp_validate_graph found a violated precondition */
} eqmp_status;

typedef enum { EQMP_F32 = 0, EQMP_BF16 = 1 } eqmp_dtype;

/*
 * Per-path channel weights.  Exactly one of the two modes:
 *   shared:  w != NULL, R == M == NULL, K == 0.
 *            w[34][C] fp32, path-major: W[e,p,c] = w[p*C + c] for every edge.
 *   radial:  w == NULL, K == 8, R and M non-NULL (may be NULL when E == 0).
 *            R[E][K] fp32 (per-edge radial features, row e = absolute edge
 *            index, 16-byte aligned), M[K][34*C] fp32 (column p*C + c,
 *            16-byte aligned): W[e,p,c] = sum_k R[e*K+k] * M[k*34*C + p*C + c].
 */
typedef struct {
  const float* w;
  const float* R;
  const float* M;
  int32_t K;
} eqmp_weights;

/* Number of CG paths (34). */
int32_t eqmp_num_paths(void);

/* Writes the (l1, l2, l3) of each path, path-major, into HOST l1l2l3[34*3].
 * EQMP_ERR_INVALID_ARG if l1l2l3 is NULL. */
eqmp_status eqmp_path_table(int32_t* l1l2l3);

/* Static, human-readable name of a status code (never NULL). */
const char* eqmp_status_string(eqmp_status s);

/*
 * Real spherical harmonics of each edge vector (Batmobile blog, section
 * "2. 寄存器中间计算"): Y[e][k] for vec[e][0..2], k = l*l+l+m.
 *   vec  [E][3] fp32, 4-byte aligned;  Y [E][16] fp32, 16-byte aligned.
 *   E >= 0 (E == 0 launches nothing).
 */
eqmp_status eqmp_sh(const float* vec, int64_t E, float* Y, eqmp_stream_t stream);

/*
 * CG tensor product + receiver sum with the harmonics read from memory
 * (the unfused second and third steps; Batmobile blog, sections
 * "1. 编译时常量" and "3. 操作融合").
 *   Y            [E][16] fp32 (e.g. from eqmp_sh), 16-byte aligned
 *   x            [N_src][C][16], x_dtype (fp32 or bf16), 16-byte aligned
 *   row_offsets  [N+1] int32, absolute edge indices (see above)
 *   src          [E] int32 sender of each edge
 *   N            receivers (rows of out), N >= 0;  E edges, 0 <= E < 2^31
 *   C            channels, one of 8, 16, 32, 64, 128
 *   weights      shared or radial, see eqmp_weights
 *   out          [N][C][16], out_dtype == x_dtype, 16-byte aligned
 */
eqmp_status eqmp_tp_scatter(const float* Y, const void* x, int64_t N_src, eqmp_dtype x_dtype,
                            const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                            int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                            eqmp_stream_t stream);

/*
 * The fused layer: SH in registers + CG tensor product + receiver sum in one
 * kernel, each edge vector read once and each output row written once
 * (Batmobile blog, section "3. 操作融合").  Arguments as eqmp_tp_scatter,
 * with vec [E][3] fp32 (4-byte aligned) in place of Y.  With radial
 * weights it runs the aligned-frame schedule of eqmp_fused_so2 (the same
 * result; fewer FMAs when the weights change per edge).
 */
eqmp_status eqmp_fused(const float* vec, const void* x, int64_t N_src, eqmp_dtype x_dtype,
                       const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                       int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                       eqmp_stream_t stream);

/*
 * eqmp_fused for a caller whose inputs and result live in host memory: one
 * call stages a whole step on `stream`, in this order:
 *   1. a copy of in_bytes bytes from h_in (host) to d_in (device);
 *   2. eqmp_fused with the layer arguments given, device pointers that may
 *      point into d_in (the caller packs the step's arrays into one block);
 *   3. a copy of out_bytes bytes from out (device) to h_out (host).
 * The caller synchronises `stream` before reading h_out.  h_in and h_out
 * should be page-locked for the copies to overlap the host; pageable memory
 * works, with copies that wait for the host.  No device memory is
 * allocated.
 *   h_in, d_in   host / device blocks of in_bytes bytes (NULL only with
 *                in_bytes == 0)
 *   h_out        host block of out_bytes bytes (NULL only with
 *                out_bytes == 0); out_bytes <= the size of out
 * Errors: EQMP_ERR_INVALID_ARG for a missing block or out_bytes beyond out,
 * before any copy; the layer's errors as eqmp_fused (the input copy is then
 * already queued, the output copy is not); EQMP_ERR_CUDA when a copy cannot
 * be queued.
 */
eqmp_status eqmp_fused_staged(const void* h_in, void* d_in, size_t in_bytes, const float* vec,
                              const void* x, int64_t N_src, eqmp_dtype x_dtype,
                              const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                              int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                              void* h_out, size_t out_bytes, eqmp_stream_t stream);

/*
 * A staged step recorded once and replayed: eqmp_plan_staged takes the
 * arguments of eqmp_fused_staged (without the stream), records the input
 * copy, the layer and the result copy into a CUDA graph (captured on a
 * private stream; nothing runs at this point) and returns it in *plan.
 * eqmp_plan_launch replays the whole step on `stream` with one graph
 * launch, asynchronously; the caller synchronises before reading h_out.
 * A plan keeps the pointers and sizes it was made with: the buffers must
 * stay allocated, and h_in and h_out page-locked, until it is destroyed;
 * their contents may change between launches.  Launches of one plan must
 * not overlap each other (same stream, or ordered by the caller).
 * eqmp_plan_destroy frees the graph (NULL: no-op).
 * Errors: as eqmp_fused_staged at planning time (then *plan = NULL);
 * EQMP_ERR_INVALID_ARG for a NULL plan; EQMP_ERR_CUDA when the capture,
 * instantiation or launch fails.  The plan records the layer's launch
 * configuration for the device current at planning time.
 */
typedef struct eqmp_plan_st* eqmp_plan;

eqmp_status eqmp_plan_staged(const void* h_in, void* d_in, size_t in_bytes, const float* vec,
                             const void* x, int64_t N_src, eqmp_dtype x_dtype,
                             const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                             int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                             void* h_out, size_t out_bytes, eqmp_plan* plan);
eqmp_status eqmp_plan_launch(eqmp_plan plan, eqmp_stream_t stream);
eqmp_status eqmp_plan_destroy(eqmp_plan plan);

/*
 * Backward of eqmp_fused (fp32 storage): gradients of a scalar loss L given
 * grad_out = dL/dout [N][C][16] fp32 (16-byte aligned):
 *   grad_x   [N_src][C][16]  dL/dx, every row written (0 for nodes that send nothing)
 *   grad_w   [34][C]         dL/dw            (shared weights)
 *   grad_R   [E][8]          dL/dR            (radial weights; rows of this call's edges)
 *   grad_M   [8][34*C]       dL/dM            (radial weights)
 *   grad_vec [E][3]          dL/dvec, forces through the harmonics' derivative
 *                            (rows of this call's edges; 0 for zero-length vectors)
 * Any output may be NULL to skip it.  The chain rule is the plain one (see
 * the forward formula); the harmonics' derivative is that of the real SH in
 * the blog's section "2. 寄存器中间计算", n = v/|v| projected.
 * dL/dx needs the sender-grouped view of the same edges: send_edges[E_send]
 * lists edge ids grouped by sender, send_offsets[N_src+1] indexes it, and
 * dst[E] gives each edge's receiver (0-based, < N).  The other gradients use
 * row_offsets/src like the forward.  workspace: device memory of at least
 * eqmp_fused_backward_workspace_size(N, E, C, radial) bytes (16-byte aligned),
 * used for the fixed-order (deterministic) weight-gradient reductions; its
 * contents on entry are ignored.  x must be fp32.  Nothing synchronises
 * the stream.
 */
int64_t eqmp_fused_backward_workspace_size(int64_t N, int64_t E, int32_t C, int32_t radial);

eqmp_status eqmp_fused_backward(const float* vec, const float* x, int64_t N_src,
                                const int32_t* row_offsets, const int32_t* src, const int32_t* dst,
                                const int32_t* send_offsets, const int32_t* send_edges, int64_t E_send,
                                int64_t N, int64_t E, int32_t C, eqmp_weights weights,
                                const float* grad_out, float* grad_x, float* grad_w, float* grad_R,
                                float* grad_M, float* grad_vec, void* workspace, int64_t workspace_bytes,
                                eqmp_stream_t stream);

/*
 * eqmp_fused_backward without a workspace argument: for callers that cannot
 * give the library extra device memory, such as a plugin inside a framework
 * that owns the whole device memory pool, or a simulation loop that must not
 * allocate on every step.  (The pages have no counterpart; this is a
 * deployment variant of eqmp_fused_backward.)  Arguments and results are
 * those of eqmp_fused_backward minus workspace/workspace_bytes.
 *   - It allocates nothing.  Its scratch is one static device array of
 *     eqmp_fused_backward_noalloc_max_bytes() bytes (8 MiB), held by every
 *     GPU that loads the library until the process exits.
 *   - The first call on a device looks up the array's device address (once
 *     per device, on the current device); make that first call before any
 *     stream capture.
 *   - Shared weights: any size (the weight-gradient reduction uses fewer,
 *     larger partial blocks so its partials fit the array).  Radial weights:
 *     E * 34 * C * 4 bytes must fit the array when grad_vec, grad_R or grad_M
 *     is requested, else EQMP_ERR_UNSUPPORTED (use eqmp_fused_backward).
 *   - All calls share the array, which keeps the previous call's contents;
 *     every part a call reads is written first by that call.  Calls that
 *     overlap on the GPU (other streams or threads) race on the array.
 */
int64_t eqmp_fused_backward_noalloc_max_bytes(void);

eqmp_status eqmp_fused_backward_noalloc(const float* vec, const float* x, int64_t N_src,
                                        const int32_t* row_offsets, const int32_t* src, const int32_t* dst,
                                        const int32_t* send_offsets, const int32_t* send_edges,
                                        int64_t E_send, int64_t N, int64_t E, int32_t C,
                                        eqmp_weights weights, const float* grad_out, float* grad_x,
                                        float* grad_w, float* grad_R, float* grad_M, float* grad_vec,
                                        eqmp_stream_t stream);

/*
 * The same layer as eqmp_fused, computed per edge in the aligned frame of
 * E2Former-V2 section 2.1 (EAAS): the sender features are rotated into a
 * frame whose z axis is the edge (Wigner-D blocks of the frame rotation),
 * where the edge harmonics keep only m = 0 (Lemma 4.1) and each output order
 * takes one input order (Eq. 13, 111 terms instead of 611), then rotated
 * back and summed into the receiver.  Exact up to rounding; about 2.5x fewer
 * FMAs per edge and channel, so it is the faster choice for per-edge
 * (radial) weights.  Arguments and results as eqmp_fused.  Launched in
 * clusters of two CTAs that may sum one receiver in two pieces (added in
 * a fixed order, so results stay bitwise reproducible on one device).
 */
eqmp_status eqmp_fused_so2(const float* vec, const void* x, int64_t N_src, eqmp_dtype x_dtype,
                           const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                           int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                           eqmp_stream_t stream);

/*
 * The fused layer at degree l_max = 4, 5 or 6 (the Batmobile blog stops at
 * l <= 3 and names higher degrees as future work).  Same definition as
 * eqmp_fused with every path (l1, l2, l3), all <= l_max, in the order
 * l1 = 0..l_max, l2 = 0..l_max, l3 = |l1-l2|..min(l_max, l1+l2)
 * (eqmp_num_paths_lmax: 65, 111, 175 paths), components k = l*l + l + m.
 * Computed in the aligned frame of E2Former-V2 section 2.1 (Lemma 4.1,
 * Eq. 13: O(l^3) terms per edge instead of the dense O(l^6)); exact up to
 * rounding.
 *   x    [N_src][C][(l_max+1)^2] fp32, 16-byte aligned (rows are bulk-copied);
 *        out [N][C][(l_max+1)^2] fp32, written
 *   weights  shared w[P][C], or radial R[E][8] (16-byte aligned), M[8][P*C]
 *   other arguments as eqmp_fused; C in {8, 16, 32, 64, 128}.
 * EQMP_ERR_UNSUPPORTED for other l_max (l_max = 3 is eqmp_fused).
 */
int32_t eqmp_num_paths_lmax(int32_t l_max);

eqmp_status eqmp_fused_lmax(int32_t l_max, const float* vec, const float* x, int64_t N_src,
                            const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                            int32_t C, eqmp_weights weights, float* out, eqmp_stream_t stream);

/*
 * Radius graph: the step before the layer.  E2Former-V2 (section 4.2,
 * deployment notes) builds neighbour lists by a radius cutoff instead of a
 * fixed k nearest neighbours; the Batmobile blog (monitoring section) takes
 * the cutoff as 4-6 Angstrom.  Open boundaries (no periodic images).
 *
 * Edges: sender j -> receiver i for every ordered pair i != j with
 * d2 < cutoff*cutoff, where, in float32 with each operation rounded on its
 * own, d_a = pos[j][a] - pos[i][a] and d2 = (d_x*d_x + d_y*d_y) + d_z*d_z.
 * The result is bitwise deterministic and independent of the hardware's
 * scheduling.
 *
 *   pos          [N][3] fp32, device.  |pos| / cutoff < about 4096 per
 *                coordinate and finite, else *E_total = -1 and the other
 *                outputs are unspecified.
 *   cutoff       > 0, finite (EQMP_ERR_INVALID_ARG otherwise).
 *   row_offsets  [N+1] int32, device, written: CSR rows by receiver,
 *                row_offsets[0] = 0, row_offsets[N] = E.
 *   src          [E_cap] int32, device, written: senders, ascending in a row.
 *   vec          [E_cap][3] fp32, device, written: pos[src] - pos[receiver]
 *                (one float32 subtraction per component).
 *   dst          [E_cap] int32 or NULL: receiver of each edge.
 *   rev          [E_cap] int32 or NULL: index of the reverse edge
 *                (receiver <- sender).  For this symmetric relation
 *                (row_offsets, rev) is the sender view that
 *                eqmp_fused_backward takes as (send_offsets, send_edges).
 *   E_cap        capacity of src/vec/dst/rev in edges (>= 0).
 *   E_total      one int64 in device memory, written with E, or -1 (bad
 *                positions) or -2 (E >= 2^31).  If E > E_cap, row_offsets is
 *                still valid but src/vec/dst/rev are unspecified: allocate
 *                E edges and call again.
 *   workspace    device memory, 256-byte aligned, of at least
 *                eqmp_radius_graph_workspace_size(N) bytes (40 to 56 N
 *                bytes, plus 384 N bytes of per-row scratch for
 *                N <= 2^21); owned by the caller; no other call may use it
 *                until this one completes.
 * N up to 2^30 (EQMP_ERR_UNSUPPORTED above).  Asynchronous on `stream`; no
 * host synchronisation.  Cost is linear in N for bounded density; a row
 * longer than 512 edges is sorted in time quadratic in its length.
 */
size_t eqmp_radius_graph_workspace_size(int64_t N);

eqmp_status eqmp_radius_graph(const float* pos, int64_t N, float cutoff, int32_t* row_offsets,
                              int32_t* src, float* vec, int32_t* dst, int32_t* rev, int64_t E_cap,
                              int64_t* E_total, void* workspace, size_t workspace_bytes,
                              eqmp_stream_t stream);

/*
 * Radius graph with periodic boundaries.  E2Former-V2 (section 4.2) treats
 * periodic systems by expanding the cells, one image per direction.  The box
 * is orthorhombic with sides box_lengths[0..2] (host memory, > 0, finite,
 * else EQMP_ERR_INVALID_ARG), the atoms lie inside it, and the cutoff is at
 * most the smallest side (EQMP_ERR_UNSUPPORTED otherwise), so that one image
 * per direction holds every neighbour.
 *
 * Edges: (sender j, image s) -> receiver i for every s in {-1, 0, 1}^3 and
 * every j with d2 < cutoff*cutoff, except j = i with s = 0, where, in
 * float32 with each operation rounded on its own,
 * d_a = (pos[j][a] - pos[i][a]) + s_a * box_lengths[a] (s_a * L_a is exact)
 * and d2 = (d_x*d_x + d_y*d_y) + d_z*d_z.  A sender may appear in a row
 * several times, once per image in reach (cutoff > L/2).  With s = 0 the
 * arithmetic is that of eqmp_radius_graph, bit for bit.
 *
 *   pos          [N][3] fp32, device; 0 <= pos[i][a] < box_lengths[a], else
 *                *E_total = -1 and the other outputs are unspecified.
 *   img          [E_cap] int32, device, written (required when E_cap > 0):
 *                image index sigma = (s_x+1) + 3 (s_y+1) + 9 (s_z+1) of
 *                each edge (13 is s = 0).  Rows are sorted by sender, then
 *                sigma.
 *   vec          [E_cap][3] fp32, device, written: d above.
 *   rev          [E_cap] int32 or NULL: index of the reverse edge, which is
 *                (receiver <- sender) with the opposite image, 26 - sigma.
 *   other arguments, E_total, the capacity protocol and the workspace
 *                (eqmp_radius_graph_workspace_size(N) bytes): as
 *                eqmp_radius_graph.
 * N up to 2^26 (EQMP_ERR_UNSUPPORTED above).  Asynchronous on `stream`.
 */
eqmp_status eqmp_radius_graph_pbc(const float* pos, int64_t N, float cutoff, const float* box_lengths,
                                  int32_t* row_offsets, int32_t* src, float* vec, int32_t* img,
                                  int32_t* dst, int32_t* rev, int64_t E_cap, int64_t* E_total,
                                  void* workspace, size_t workspace_bytes, eqmp_stream_t stream);

/*
 * Synchronous check of the graph preconditions on device data:
 * 0 <= row_offsets[0] <= ... <= row_offsets[N] <= E and
 * 0 <= src[e] < N_src for every e in [row_offsets[0], row_offsets[N]).
 * Returns EQMP_OK or EQMP_ERR_GRAPH (or an argument/CUDA error).  Runs a
 * small kernel on `stream` and waits for it.
 */
eqmp_status eqmp_validate_graph(const int32_t* row_offsets, const int32_t* src, int64_t N,
                                int64_t N_src, int64_t E, eqmp_stream_t stream);

/*
 * Reads and clears the current device's watchdog word (synchronises the
 * device).  *code = 0 when no bounded wait has given up since the last
 * call; otherwise a nonzero code naming the wait: 1 a consumer waiting for
 * a gathered row, 2 a producer waiting for a free slot, 3 a producer
 * draining its last slots, 4 a grid barrier of eqmp_radius_graph, 5 the
 * self-test below, 7 the look-back of eqmp_radius_graph's prefix sums,
 * 8 a CTA of the aligned-frame layer waiting for the piece of a receiver
 * that the next CTA of its cluster summed.
 * A nonzero code means the outputs of the kernels since the last call are
 * unspecified.  Returns
 * EQMP_ERR_DEVICE_TIMEOUT when *code != 0.
 */
eqmp_status eqmp_device_error(int32_t* code);

/*
 * Self-test of the failure reporting above: launches one thread that waits
 * on a barrier nothing completes, with a limit of wait_ms milliseconds
 * (1..1000, else EQMP_ERR_INVALID_ARG).  The wait gives up and records
 * code 5; the next eqmp_device_error returns EQMP_ERR_DEVICE_TIMEOUT with
 * *code = 5, and the device stays usable.  Nothing faults or hangs.
 */
eqmp_status eqmp_watchdog_selftest(int32_t wait_ms, eqmp_stream_t stream);

/* FP32 throughput probe: the denominator of the layer kernels' roofline.
 * Launches `blocks_per_sm` x (SM count) CTAs of 256 threads; each thread runs
 * `iters` rounds of 8 independent paired FP32 FMAs (fma.rn.f32x2), i.e.
 * 32 * iters flops per thread, nothing else but a final conditional store.
 * The caller times the launch (CUDA events on `stream`) and divides.
 * `out`: device pointer to one float; written only if the sums reach a value
 * they never reach (it keeps the arithmetic from being removed).
 * Writes the launch's flop count to *flops (host pointer).
 * Errors: EQMP_ERR_INVALID_ARG for a null pointer, iters < 1 or
 * blocks_per_sm outside [1, 8]; EQMP_ERR_CUDA for a failed launch. */
eqmp_status eqmp_fp32_peak_probe(int32_t iters, int32_t blocks_per_sm, float* out, double* flops,
                                 eqmp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EQMP_H */
