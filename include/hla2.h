/*
 * hla2.h -- C ABI of libhla2: masked second-order Higher-order Linear
 * Attention (HLA) on NVIDIA GB300 (sm_103a).
 *
 * Source of the method: the technical summary pages of "Higher-order Linear
 * Attention" (arXiv 2510.27258), Japanese and French editions (gist.science),
 * cited below as [HLA §1] ("Second-order HLA"), [HLA §2] ("AHLA"), [HLA §4]
 * ("Parallel training via associative scans") and [HLA R] ("Results and
 * claims").
 *
 * Per head, with tokens t = 0..T-1, q_t, k_t in R^d and v_t in R^dv:
 *   S_t = sum_{i<=t} k_i k_i^T      C_t = sum_{i<=t} q_i v_i^T     m_t = sum_{i<=t} q_i
 *   G_t = G_{t-1} + k_t k_t^T C_{t-1}          h_t = h_{t-1} + k_t k_t^T m_{t-1}
 *   o_t = q_t^T (S_t C_t - G_t) = sum_{i<=j<=t} (q_t.k_i)(k_i.q_j) v_j        [HLA §1]
 *   ratio-normalised: o_t / (q_t^T (S_t m_t - h_t))                            [HLA §1]
 * (The pages name G_t and h_t without printing their update; the update above
 * is the reading that makes o_t the causal sum, and it is what this library
 * computes.)
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers, owned by the caller.  The
 *    library never allocates, frees or keeps them past the call.
 *  - Tensors are dense, row-major, with no padding:
 *      Q, K: [B][H][T][d]     V: [B][H][T][dv]     O: [B][H][T][dv] (fp32)
 *    and every pointer must be 16-byte aligned.
 *  - `dtype` gives the element type of Q, K, V: HLA2_DTYPE_F32 (float) or
 *    HLA2_DTYPE_BF16 (bfloat16).  All arithmetic accumulates in fp32.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronising, except
 *    hla2_device_status.
 *  - Return value: HLA2_OK (0) or a negative HLA2_ERR_* code; a one-line
 *    reason is kept per host thread for hla2_last_error_detail.
 *  - T need not be a multiple of any chunk length: the ragged tail behaves as
 *    if padded with zero tokens, which leaves every output unchanged.
 *  - Supported sizes: 1 <= d, dv <= 128 and B*H <= 65535 for the forward,
 *    summary and scan calls; d, dv powers of two in [4, 128] for hla2_step.
 */
#ifndef HLA2_H
#define HLA2_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define HLA2_API __attribute__((visibility("default")))
#else
#define HLA2_API
#endif

/* ABI-compatible with cudaStream_t without including CUDA headers. */
typedef struct CUstream_st* hla2_stream_t;

enum {
    HLA2_OK = 0,
    HLA2_ERR_INVALID = -1,     /* null pointer, misaligned pointer, non-positive size */
    HLA2_ERR_UNSUPPORTED = -2, /* size or type outside what this build supports */
    HLA2_ERR_WORKSPACE = -3,   /* workspace pointer null or smaller than required */
    HLA2_ERR_LAUNCH = -4,      /* a CUDA call or kernel launch failed */
    HLA2_ERR_DEVICE = -5       /* a kernel reported a device-side error (timeout, bounds) */
};

enum { HLA2_DTYPE_F32 = 0, HLA2_DTYPE_BF16 = 1 };

/*
 * Bytes of device workspace hla2_forward needs for this problem (valid for
 * either value of `normalized`).  Returns 0 for sizes hla2_forward rejects.
 * The size depends on the segment plan, which depends on the SM count of the
 * CURRENT device: query it with the device that will run the forward current
 * (without a visible device the plan assumes 152 SMs).
 */
HLA2_API size_t hla2_forward_workspace(int B, int H, int T, int d, int dv, int dtype);

/*
 * The forward's segment plan [HLA §4: the sequence is cut into segments
 * whose summaries are scanned]: each head's ceil(T/128) chunks of 128 tokens
 * are cut into *nseg runs of *chunks_per_segment chunks (the last run may be
 * shorter), one CTA per run.  sm_count > 0 plans for that many SMs (what-if
 * queries, tests); sm_count <= 0 uses the current device's SM count, which is
 * what hla2_forward does.  *sm_count_used (may be NULL) receives the count
 * planned for.  Host only: reads the device attribute once per device, no
 * GPU work.  Errors: HLA2_ERR_INVALID (B, H, T <= 0 or a NULL nseg /
 * chunks_per_segment), HLA2_ERR_UNSUPPORTED (B*H > 65535).
 */
HLA2_API int hla2_forward_plan(int B, int H, int T, int sm_count, int* nseg, int* chunks_per_segment,
                               int* sm_count_used);

/*
 * Masked second-order HLA forward, chunk-parallel [HLA §4]: the sequence of
 * each head is cut into segments; every segment's summary is computed in
 * parallel, an exclusive scan with the semidirect-product combine gives each
 * segment its prefix state, and every segment then walks its chunks from that
 * prefix, emitting o_t.  The result equals the serial recurrence [HLA §1]
 * up to fp32 rounding [HLA §4].
 *
 *   Q, K, V   inputs as above (dtype), read only.
 *   O         [B][H][T][dv] fp32 output, fully overwritten.
 *   normalized  0: o_t as above; 1: ratio-normalised o_t (plain IEEE division,
 *             a zero denominator gives inf/NaN).
 *   workspace device scratch of at least hla2_forward_workspace(...) bytes,
 *             16-byte aligned; contents need not be initialised and are
 *             garbage afterwards.
 *   state_out optional (NULL to skip): receives each head's final state after
 *             token T-1 in the hla2_step layout, [B*H][d*d + 2*d*dv + 2*d]
 *             fp32, so that decoding can continue with hla2_step.  On the
 *             tensor-core path (hla2_forward_path == 1) its G part carries the
 *             outputs' bf16-operand rounding; S, C and m are fp32 sums.
 * Errors: HLA2_ERR_INVALID (nulls, sizes <= 0, misalignment),
 *         HLA2_ERR_UNSUPPORTED (d or dv > 128, unknown dtype),
 *         HLA2_ERR_WORKSPACE, HLA2_ERR_LAUNCH.
 */
HLA2_API int hla2_forward(const void* Q, const void* K, const void* V, float* O,
                 int B, int H, int T, int d, int dv, int normalized, int dtype,
                 void* workspace, size_t ws_bytes, float* state_out, hla2_stream_t stream);

/*
 * hla2_forward without a caller workspace.  The pages have no counterpart to
 * this call; it exists for callers that cannot allocate device memory where
 * they run the forward (a host framework that owns a fixed device arena and
 * bans cudaMalloc from its callbacks, a runtime that hands its plugins only
 * input and output buffers, a loop where allocation is forbidden after
 * start-up).  It computes exactly what hla2_forward computes with
 * state_out = NULL, taking its scratch from a fixed 64 MiB array that the
 * library defines as a static device object: every GPU that loads the
 * library holds that array until the process exits.
 *  - Problems whose hla2_forward_workspace(...) exceeds 64 MiB are rejected
 *    with HLA2_ERR_UNSUPPORTED and a message saying so; nothing runs.
 *  - The first call made on a device (with it current) looks up the array's
 *    device address; make that first call before any stream capture.
 *  - All calls share the array and it keeps the previous call's contents
 *    (nothing in it needs to start at zero).  Calls whose GPU work overlaps,
 *    e.g. on two streams, race on it: the caller must serialise them.
 *  - No cudaMalloc, cudaFree or allocating library routine is called.
 * Other arguments and errors as for hla2_forward.
 */
HLA2_API int hla2_forward_noalloc(const void* Q, const void* K, const void* V, float* O,
                                  int B, int H, int T, int d, int dv, int normalized, int dtype,
                                  hla2_stream_t stream);

/*
 * The forward on HOST buffers: the masked operator of hla2_forward, with the
 * copies in and out made by the library.  The pages have no counterpart (it
 * is the end-to-end entry point).  Heads are independent, so the B*H heads
 * are cut into groups of heads_per_group (0: about an eighth of them) and
 * each group's host-to-device copy of Q, K, V, its forward and the
 * device-to-host copy of its O run as a pipeline: the copy of one group
 * overlaps the forward of the previous one and the copy-out of the one
 * before.  The copies run on two streams the library creates once per device
 * and keeps (with eight events); the forwards run on `stream`, which, when
 * the call returns, carries all of the call's work: O is complete once
 * `stream` has been synchronised.
 *   Qh, Kh [B][H][T][d], Vh [B][H][T][dv] on the host in `dtype`, Oh
 *   [B][H][T][dv] fp32 on the host.  They should be page-locked (pinned):
 *   copies from pageable memory run, but without overlap.
 *   dev: device buffer of hla2_forward_host_workspace(...) bytes, 256-byte
 *   aligned, owned by the caller: two slots of a group's Q, K, V, O and one
 *   forward workspace.
 * Results equal hla2_forward's within its tolerances (each group is planned
 * as its own problem, so segment boundaries, and with them rounding, can
 * differ).  Calls on one device enqueue one at a time (a lock); their copies
 * share the library's two copy streams.  Errors as for hla2_forward, plus
 * HLA2_ERR_WORKSPACE for a missing or small `dev`; work enqueued before an
 * error is left on the streams.
 */
HLA2_API size_t hla2_forward_host_workspace(int B, int H, int T, int d, int dv, int dtype, int heads_per_group);
HLA2_API int hla2_forward_host(const void* Qh, const void* Kh, const void* Vh, float* Oh,
                               int B, int H, int T, int d, int dv, int normalized, int dtype,
                               int heads_per_group, void* dev, size_t dev_bytes, hla2_stream_t stream);

/*
 * One streaming decode step for n independent heads [HLA §1, online update;
 * HLA R: O(d^2 + d dv) per token, independent of the prefix length].
 *   state  [n][d*d + 2*d*dv + 2*d] fp32, per head S (d x d) | C (d x dv) |
 *          G (d x dv) | m (d) | h (d), row-major; read and updated in place.
 *   q, k   [n][d] fp32;  v [n][dv] fp32;  o [n][dv] fp32 output.
 *   The token is absorbed first (G += k k^T C, h += k k^T m, then S, C, m
 *   grow), then o = q^T (S C - G) is emitted (divided by q^T (S m - h) when
 *   normalized).  A zero state is the empty prefix.
 * Errors: HLA2_ERR_INVALID, HLA2_ERR_UNSUPPORTED (d or dv not a power of two
 *         in [4, 128]), HLA2_ERR_LAUNCH.
 */
HLA2_API int hla2_step(float* state, const float* q, const float* k, const float* v, float* o,
              int n, int d, int dv, int normalized, hla2_stream_t stream);

/*
 * hla2_step on the compact "P-form" decode state [HLA §1 online update,
 * rewritten with P = S C - G and p = S m - h]:
 *   state  [n][d*d + d*dv + d] fp32, per head S (d x d) | P (d x dv) | p (d).
 * The step computes S' = S + k k^T, u = S' q, o = q^T P + (q.u) v,
 * P' = P + u v^T, p' = p + u (normalised: o /= q.p'), i.e. the same o_t as
 * hla2_step, moving a third fewer state bytes at d = dv.  Same argument
 * rules and errors as hla2_step; a zero state is the empty prefix.
 */
HLA2_API int hla2_step_pform(float* state, const float* q, const float* k, const float* v, float* o,
                             int n, int d, int dv, int normalized, hla2_stream_t stream);

/*
 * Converts n decode states from the hla2_step layout S|C|G|m|h to the P-form
 * layout S|P|p (P = S C - G, p = S m - h, fp32 products).  gstate and
 * pstate must not overlap.  Errors as for hla2_step (d, dv <= 128).
 */
HLA2_API int hla2_state_to_pform(const float* gstate, float* pstate, int n, int d, int dv,
                                 hla2_stream_t stream);

/*
 * Summary of every chunk of L consecutive tokens [HLA §4, segment summaries]:
 * the state the recurrence of [HLA §1] reaches from zero on that chunk alone.
 *   summ  [B][H][N][d*d + 2*d*dv + 2*d] fp32, N = ceil(T/L), record
 *         S (d x d) | C (d x dv) | m (d) | G (d x dv) | h (d).
 *         The last chunk may be shorter than L.
 * Errors: HLA2_ERR_INVALID, HLA2_ERR_UNSUPPORTED, HLA2_ERR_LAUNCH.
 */
HLA2_API int hla2_chunk_summaries(const void* Q, const void* K, const void* V, float* summ,
                         int B, int H, int T, int d, int dv, int L, int dtype,
                         hla2_stream_t stream);

/*
 * Exclusive scan over N summaries per head with the semidirect-product
 * combine of [HLA §4] (A earlier, B later):
 *   S = S_A + S_B, C = C_A + C_B, m = m_A + m_B,
 *   G = G_A + G_B + S_B C_A,  h = h_A + h_B + S_B m_A.
 * prefix[n] = summ[0] o ... o summ[n-1], prefix[0] = zero (the identity).
 *   summ, prefix  [B][H][N][record] as for hla2_chunk_summaries; must not
 *                 overlap.
 * Because S, C and m combine by plain addition, the scan is evaluated as an
 * exclusive sum of (S, C, m), one product S_r C_<r (and S_r m_<r) per record,
 * and an exclusive sum of G_r + S_r C_<r: the same value as any bracketing of
 * the combine, up to fp32 rounding.  With d = dv in {64, 128} on sm_103 the
 * products S_r C_<r run on the tensor cores with each fp32 operand split into
 * bf16 hi + lo parts (about 16 significant bits per operand, fp32
 * accumulation); S_r m_<r and every sum stay fp32 on the CUDA cores.
 * Errors: HLA2_ERR_INVALID, HLA2_ERR_UNSUPPORTED, HLA2_ERR_LAUNCH.
 */
HLA2_API int hla2_scan(const float* summ, float* prefix, int B, int H, int N, int d, int dv,
              hla2_stream_t stream);

/*
 * AHLA, the asymmetric second-order variant [HLA §2]: the operator
 * Q (K^T Q)(K^T V) with streaming summaries P^KV, m^K, E, n.  Under the
 * causal mask (the reading this library computes; the pages print no update)
 *   o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j            (A A V, A = tril(Q K^T))
 *   P_t = P_{t-1} + k_t v_t^T      m_t = m_{t-1} + k_t
 *   E_t = E_{t-1} + k_t (P_t^T q_t)^T      n_t = n_{t-1} + k_t (q_t . m_t)
 *   o_t = E_t^T q_t;  ratio-normalised: o_t / (q_t . n_t).
 * The forward runs like hla2_forward [HLA §4]: segment summaries
 * M|P|m|E|n (M = sum k q^T, needed only to join segments), an exclusive scan
 * with the combine E = E_A + E_B + M_B P_A, n = n_A + n_B + M_B m_A (HLA's
 * combine with S -> M, C -> P, G -> E, h -> n), then segment walks from the
 * prefixes.  Arguments, layouts, workspace (hla2_forward_workspace) and
 * errors as for hla2_forward, except state_out:
 *   state_out optional: [B*H][2*d*dv + 2*d] fp32, per head
 *             P (d x dv) | E (d x dv) | m (d) | n (d), the hla2_ahla_step layout.
 */
HLA2_API int hla2_ahla_forward(const void* Q, const void* K, const void* V, float* O,
                               int B, int H, int T, int d, int dv, int normalized, int dtype,
                               void* workspace, size_t ws_bytes, float* state_out, hla2_stream_t stream);

/*
 * Which implementation hla2_ahla_forward picks on the current device:
 * 1 = tensor-core segment walks (tcgen05; bf16 d = dv in {64, 128},
 * unnormalised, no state_out), 0 = CUDA-core segment walks (fp32).
 */
HLA2_API int hla2_ahla_forward_path(int d, int dv, int dtype, int normalized, int with_state_out);

/*
 * One AHLA decode step for n heads [HLA §2 streaming summaries].
 *   state  [n][2*d*dv + 2*d] fp32, per head P | E | m | n, updated in place;
 *          a zero state is the empty prefix.
 *   q, k [n][d], v [n][dv], o [n][dv], all fp32.
 * The token is absorbed (P, m first, then E, n), then o = E^T q is emitted
 * (divided by q.n when normalized).  Same size rules and errors as hla2_step.
 */
HLA2_API int hla2_ahla_step(float* state, const float* q, const float* k, const float* v, float* o,
                            int n, int d, int dv, int normalized, hla2_stream_t stream);

/*
 * Unmasked second-order operator [HLA §1: S_t C_t is the naive product that
 * G_t corrects; HLA R lists the unmasked operator as a variant]:
 *   o_t = q_t^T S_t C_t = sum_{i<=t, j<=t} (q_t.k_i)(k_i.q_j) v_j,
 *   ratio-normalised: o_t / (q_t^T S_t m_t).
 * Segments carry only S, C, m, which join by plain addition, so the scan is a
 * running sum [HLA §4 with no cross term].  Arguments, layouts, workspace
 * (hla2_forward_workspace) and errors as for hla2_forward, except state_out:
 *   state_out optional: [B*H][d*d + d*dv + d] fp32, per head S | C | m, the
 *             hla2_unmasked_step layout.
 * Implementation: see hla2_unmasked_forward_path.
 */
HLA2_API int hla2_unmasked_forward(const void* Q, const void* K, const void* V, float* O,
                                   int B, int H, int T, int d, int dv, int normalized, int dtype,
                                   void* workspace, size_t ws_bytes, float* state_out, hla2_stream_t stream);

/*
 * Which implementation hla2_unmasked_forward picks on the current device:
 * 1 = tensor-core segment walks (tcgen05 with fp32 accumulators; bf16
 * d = dv in {64, 128}, unnormalised, no state_out), 0 = CUDA-core segment
 * walks (fp32 arithmetic).
 */
HLA2_API int hla2_unmasked_forward_path(int d, int dv, int dtype, int normalized, int with_state_out);

/*
 * One decode step of the unmasked operator for n heads.
 *   state  [n][d*d + d*dv + d] fp32, per head S | C | m, updated in place.
 * S, C, m grow by the token first, then o = (S q)^T C is emitted (divided by
 * (S q) . m when normalized).  Same size rules and errors as hla2_step.
 */
HLA2_API int hla2_unmasked_step(float* state, const float* q, const float* k, const float* v, float* o,
                                int n, int d, int dv, int normalized, hla2_stream_t stream);

/*
 * Exponentially decayed masked operator.  [HLA §4] names decayed operators
 * among those the scan covers but prints no form; the reading this library
 * computes decays every prefix moment by one scalar gamma per token:
 *   S_t = gamma S + k k^T,  C_t = gamma C + q v^T,  m_t = gamma m + q,
 *   G_t = gamma^2 G + gamma k k^T C_{t-1},  h_t = gamma^2 h + gamma k k^T m_{t-1},
 *   o_t = q_t^T (S_t C_t - G_t) = sum_{i<=j<=t} gamma^{2t-i-j} (q_t.k_i)(k_i.q_j) v_j,
 * ratio-normalised by q_t^T (S_t m_t - h_t).  gamma = 1 is hla2_forward's
 * operator.  Segments join with the decayed combine (B spanning n_B tokens,
 * f = gamma^{n_B}): S = f S_A + S_B, ..., G = f^2 G_A + G_B + f S_B C_A,
 * computed as decayed running sums along the segment axis with one cross
 * product per segment.  Implementation: see hla2_decay_forward_path.
 *   gamma     in [0, 1] (else HLA2_ERR_INVALID).
 *   state_out optional: [B*H][d*d + d*dv + d] fp32, per head the compact
 *             state S | P = S C - G | p = S m - h, the hla2_decay_step layout.
 * Other arguments, workspace (hla2_forward_workspace) and errors as for
 * hla2_forward.
 */
HLA2_API int hla2_decay_forward(const void* Q, const void* K, const void* V, float* O,
                                int B, int H, int T, int d, int dv, int normalized, float gamma, int dtype,
                                void* workspace, size_t ws_bytes, float* state_out, hla2_stream_t stream);

/*
 * Which implementation hla2_decay_forward picks on the current device:
 * 1 = tensor-core segment walks (tcgen05 with fp32 accumulators; bf16
 * d = dv in {64, 128}, unnormalised, no state_out, gamma in [0.8, 1]: the
 * chunk form there carries per-token factors down to gamma^{-256}, which stay
 * finite), 0 = CUDA-core segment walks (fp32 arithmetic).
 */
HLA2_API int hla2_decay_forward_path(int d, int dv, int dtype, int normalized, int with_state_out, float gamma);

/*
 * One decayed decode step for n heads on the compact state
 * [n][d*d + d*dv + d] fp32 (S | P | p, updated in place):
 *   S = gamma S + k k^T, u = S q, P = gamma^2 P + u v^T, p = gamma^2 p + u,
 *   o = q^T P (divided by q . p when normalized).
 * gamma = 1 is hla2_step_pform.  Same size rules and errors as hla2_step,
 * plus HLA2_ERR_INVALID for gamma outside [0, 1].
 */
HLA2_API int hla2_decay_step(float* state, const float* q, const float* k, const float* v, float* o,
                             int n, int d, int dv, int normalized, float gamma, hla2_stream_t stream);

/*
 * Copies the calling host thread's last error reason (NUL-terminated,
 * truncated to n bytes) into buf.  Returns the length of the full message.
 */
HLA2_API int hla2_last_error_detail(char* buf, size_t n);

/*
 * Synchronises `stream`, then reads and clears the library's device-side
 * error word (set by a kernel whose bounded wait ran out or whose bounds
 * check failed; such a kernel skips the offending access and returns).
 * Returns HLA2_OK, HLA2_ERR_DEVICE (word was set) or HLA2_ERR_LAUNCH.
 */
HLA2_API int hla2_device_status(hla2_stream_t stream);

/*
 * Exercises the device error path on purpose, without any fault (no
 * counterpart on the pages).  Launches one CTA that takes tensor memory,
 * waits on a barrier that nothing arrives on, gives up after wait_us
 * microseconds the way every bounded wait of the library does (it sets the
 * device status word), releases its tensor memory and returns.
 *   flag     device int (caller-owned, 4-byte aligned): receives 0 when the
 *            wait gave up (1 would mean it completed, which cannot happen).
 *   wait_us  1 .. 2,000,000.
 * A following hla2_device_status returns HLA2_ERR_DEVICE (and clears the
 * word); the context stays usable.  Errors: HLA2_ERR_INVALID (null or
 * misaligned flag, wait_us out of range), HLA2_ERR_UNSUPPORTED (a device
 * without tensor memory), HLA2_ERR_LAUNCH.
 */
HLA2_API int hla2_selftest_wait_runout(int* flag, int wait_us, hla2_stream_t stream);

/*
 * Instrumentation (no counterpart on the pages).  While enabled, every
 * hla2_forward records CUDA events on its stream around its three phases:
 * [0] segment summaries, [1] exclusive scan, [2] segment outputs.
 * The library also counts every kernel it launches, enabled or not.
 */
HLA2_API int hla2_profile_enable(int on);

/*
 * Which implementation hla2_forward picks for these arguments on the current
 * device: 1 = tensor-core segment walks (tcgen05, bf16 operands, fp32
 * accumulation), 0 = CUDA-core segment walks (fp32 arithmetic).  Both are
 * CUDA kernels of this library.
 */
HLA2_API int hla2_forward_path(int d, int dv, int dtype, int normalized, int with_state_out);

/*
 * 1 when hla2_chunk_summaries with these sizes runs on the tensor cores of
 * the current device (bf16, d = dv in {64, 128}, L in {64, 128}; G and h
 * from split-bf16 operands, about 16 significant bits), 0 when it runs on
 * the fp32 CUDA-core walk.  Host only.
 */
HLA2_API int hla2_chunk_summaries_path(int d, int dv, int L, int dtype);

/*
 * Waits for the events recorded since the previous read, writes the summed
 * phase durations in milliseconds to ms_out[0..min(n,3)-1], the number of
 * profiled forwards to *forwards (if not NULL) and the number of kernels the
 * library launched since the previous read to *launches (if not NULL), then
 * clears both records.  Returns HLA2_OK or HLA2_ERR_LAUNCH.
 */
HLA2_API int hla2_profile_read(float* ms_out, int n, int* forwards, long long* launches);

#ifdef __cplusplus
}
#endif

#endif /* HLA2_H */
