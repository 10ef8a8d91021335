/*
 * libkda -- KDA (Kimi Delta Attention) layer forward on GB300 (sm_103a).
 *
 * The layer is the gated delta rule with one decay per key channel,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t,            alpha_t = exp(log_alpha_t),
 *
 * a running state of fixed size (d_k x d_v per sequence and head) as
 * described on orkas.ai, "Kimi K3 architecture" (German edition), section
 * "Sequenz: Drei Viertel der Schichten lesen nicht mehr alles".  The decay
 * is bounded below, log_alpha in [-5, 0] (each step keeps at least 0.67 % of
 * the state), so the cumulative log-decay over a 16-token tile stays in
 * [-80, 0] and its reciprocal below e^80; same page, section "Eine
 * Untergrenze, die einen GPU-Codepfad beseitigte".  That bound is what lets
 * the chunked kernels evaluate the diagonal tiles with the same dense bf16
 * tensor-core products as every other tile.
 *
 * Conventions for every entry point
 *   - All pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates or frees device memory.
 *   - Calls are asynchronous on `stream`; buffers must stay valid until the
 *     stream reaches the call.  Argument errors are returned synchronously,
 *     before anything is launched; nothing is printed and no C++ exception
 *     crosses this interface.
 *   - Layouts are row-major with the last dimension contiguous.  Activations
 *     are token-major [B, T, H, d]; states are [B or N, H, d_k, d_v] fp32.
 *   - q and k are used as given (the caller L2-normalises them).
 *   - log_alpha must lie in [-5, 0].  With KDA_CHECK_DECAY set in the
 *     environment (read once per process) the prefill entry points also
 *     scan it on the device and report a violation through
 *     kda_last_device_status(); without it, out-of-range values give
 *     unspecified results.
 *   - With KDA_ABLATE_DIAG=1 in the environment (read on every call) the
 *     prefill entry points evaluate the four diagonal 16x16 tiles of each
 *     chunk per position pair in log space on CUDA cores, the evaluation
 *     that needs no bound on the decay, instead of with the dense
 *     tensor-core products.  Results agree within rounding; it exists to
 *     measure what the bound saves.
 *   - Schedule.  kda_chunk_fwd runs a fixed-length prefill either as rounds
 *     of two kernels (an intra-chunk stage, then the state pass) or, for few
 *     (sequence, head) chains, as one cooperative launch that runs both and
 *     keeps the per-chunk records in a small ring; it picks the one measured
 *     faster for the shape.  KDA_SCHEDULE=rounds or KDA_SCHEDULE=fused in
 *     the environment (read on every call) forces one (fused where it can
 *     run: chains on at most half the SMs).  Results are the same bit for
 *     bit either way.
 *   - Supported head dims: d_k = d_v = 128, and d_k = d_v = 64 (prefill
 *     only).  Others return KDA_ERR_UNSUPPORTED.
 *   - Range.  The prefill entry points carry the state in fp32 but feed
 *     it, and the delta-rule corrections u = beta (v - S^T k) of each chunk,
 *     to the tensor cores as fp16.  State entries and corrections must stay
 *     below 6e4 in magnitude (values and states of the unit-variance kind
 *     are ~1); a larger or non-finite one sets KDA_ERR_RANGE in the device
 *     status word and the results are then unspecified.  Inside that range
 *     results scale with (v, initial_state) by powers of two.
 *   - Base pointers must be 16-byte aligned (KDA_ERR_ALIGNMENT), except
 *     beta, which needs only its natural 2-byte alignment.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifndef KDA_API
#define KDA_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad cu_seqlens on host */
    KDA_ERR_UNSUPPORTED = 2, /* head dim or dtype the library does not implement */
    KDA_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned                  */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed                 */
    KDA_ERR_DECAY_BOUND = 5, /* device found log_alpha outside [-5, 0]            */
    KDA_ERR_TIMEOUT = 6,     /* a device-side wait hit its iteration limit        */
    KDA_ERR_WORKSPACE = 7,   /* workspace missing or smaller than required        */
    KDA_ERR_RANGE = 8        /* a state-pass operand left the fp16 range          */
} kda_status_t;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype_t;

/*
 * kda_chunk_fwd -- chunked prefill of B fixed-length sequences.
 *   q, k, log_alpha : [B, T, H, d_k] bf16
 *   v               : [B, T, H, d_v] bf16
 *   beta            : [B, T, H] bf16
 *   initial_state   : [B, H, d_k, d_v] fp32, or NULL for zeros
 *   out             : [B, T, H, d_v] in out_dtype (KDA_BF16 or KDA_F32)
 *   final_state     : [B, H, d_k, d_v] fp32, or NULL (not written); may be
 *                     the same buffer as initial_state (each state is read
 *                     once before it is overwritten)
 *   scale           : multiplies every output (1.0 for the plain layer)
 *   workspace       : device scratch of at least kda_chunk_fwd_workspace_size()
 *                     bytes, 16-byte aligned, owned by the caller; it holds
 *                     the per-(chunk, head) intermediate records (65 KiB
 *                     each) passed from the intra-chunk stage to the state
 *                     pass, the fp32 state handed between segments of the
 *                     sequence, and two counters with which the intra-chunk
 *                     stage hands out its work (so calls sharing a workspace
 *                     must not overlap on the GPU).  Too small or NULL ->
 *                     KDA_ERR_WORKSPACE.
 * Long sequences run as segments of chunks, all on `stream`: the
 * intra-chunk stage of one segment is a programmatic dependent launch of
 * the previous segment's state pass and runs on the SMs that pass leaves
 * free.
 * The chunked evaluation (64-token chunks of four 16-token tiles) follows
 * the blockwise computation the orkas.ai page describes in section "Eine
 * Untergrenze, die einen GPU-Codepfad beseitigte".  out must not alias any
 * input.  T may be any value >= 0 (a partial last chunk is masked).
 */
KDA_API kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v,
                           const void* log_alpha, const void* beta,
                           const float* initial_state, void* out,
                           kda_dtype_t out_dtype, float* final_state, int B,
                           int T, int H, int d_k, int d_v, float scale,
                           void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* Bytes of device workspace kda_chunk_fwd needs for this shape:
 * R * H * 66560 + B * H * 65536 + 256 with R = B * ceil(T / 64) records per
 * head, or, for shapes that may take the segment scan (ceil(T / 64) >= 2048
 * and B * H <= 64), that of kda_chunk_fwd_segments with 8 segments when it
 * is larger.  Where one record per chunk would pass 4 GiB and the call runs
 * as overlapped segments (ceil(T / 64) >= 128 and B * H at most half the
 * SMs), the records live in a ring of two segments of at most 128 chunks
 * (R = B * 2 * segment, the ring under 1 GiB), so the size stops growing
 * with T.  The answer depends on the current device's SM count. */
KDA_API size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v);

/*
 * kda_chunk_fwd_segments -- kda_chunk_fwd with each sequence cut into
 * n_segments segments of whole 64-token chunks that are walked in parallel.
 * The serial state pass bounds a long sequence with few heads; the orkas.ai
 * page ("Kimi K3 architecture", section "Die Rechnung landet in der
 * Bereitstellungsinfrastruktur") splits a sequence by reducing each segment
 * to a cumulative transition and a zero-start state, which compose, and
 * rebuilding every segment's entry state with a prefix scan.  Here:
 *   1. the intra-chunk stage runs once over every chunk;
 *   2. segment 0 is walked from initial_state with outputs, and every later
 *      segment q twice at the same time: from zero without values' outputs
 *      (its zero-start state Z_q) and from the identity without values (its
 *      transition M_q);
 *   3. entry states E_1 = state after segment 0, E_{q+1} = M_q E_q + Z_q
 *      (fp32, one small kernel per (sequence, head));
 *   4. segments 1.. are walked again from E_q with outputs; the last one
 *      writes final_state.
 * n_segments = 1 is kda_chunk_fwd without a scan; larger values are capped
 * at 8 and at the number of chunks, and reduced so that no segment is
 * empty.  kda_chunk_fwd takes this path by itself for long sequences with
 * few (sequence, head) pairs.  Results equal kda_chunk_fwd's up to
 * rounding (the transitions are carried in fp32 through fp16 operands like
 * the state).  Arguments and results are those of kda_chunk_fwd; the
 * workspace is at least kda_chunk_fwd_segments_workspace_size() bytes.
 */
KDA_API kda_status_t kda_chunk_fwd_segments(const void* q, const void* k, const void* v,
                                            const void* log_alpha, const void* beta,
                                            const float* initial_state, void* out,
                                            kda_dtype_t out_dtype, float* final_state, int B,
                                            int T, int H, int d_k, int d_v, float scale,
                                            int n_segments, void* workspace,
                                            size_t workspace_bytes, cudaStream_t stream);
KDA_API size_t kda_chunk_fwd_segments_workspace_size(int B, int T, int H, int d_k, int d_v,
                                                     int n_segments);

/*
 * kda_chunk_fwd_checkpointed -- kda_chunk_fwd that also saves the recurrent
 * state at fixed token boundaries, for a prefix cache.  The orkas.ai page
 * ("Kimi K3 architecture", section "Die Rechnung landet in der
 * Bereitstellungsinfrastruktur") describes hashing prefixes every 512
 * tokens and keeping the fixed-size recurrent state only at a sparse subset
 * of those boundaries; this call writes it at every checkpoint_every tokens.
 *   checkpoint_every : tokens between checkpoints, a positive multiple of 64
 *                      (KDA_ERR_INVALID_ARG otherwise)
 *   checkpoints      : [B, T / checkpoint_every, H, d_k, d_v] fp32 (16-byte
 *                      aligned; may be NULL when T < checkpoint_every).
 *                      Entry [b, n] is the state after the first
 *                      (n + 1) * checkpoint_every tokens of sequence b.
 * Every other argument, the workspace size and the results are those of
 * kda_chunk_fwd.
 */
KDA_API kda_status_t kda_chunk_fwd_checkpointed(const void* q, const void* k, const void* v,
                                                const void* log_alpha, const void* beta,
                                                const float* initial_state, void* out,
                                                kda_dtype_t out_dtype, float* final_state,
                                                int B, int T, int H, int d_k, int d_v,
                                                float scale, float* checkpoints,
                                                int checkpoint_every, void* workspace,
                                                size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_chunk_fwd_host -- kda_chunk_fwd with the tensors in host memory: the
 * inputs q, k, v, log_alpha, beta and initial_state, and the outputs out and
 * final_state, are host pointers (page-locked memory for the copies to run
 * asynchronously; pageable memory works, with copies that block the calling
 * thread).  Shapes, dtypes, results and errors are those of kda_chunk_fwd,
 * without the segment scan (long sequences with few heads run as one serial
 * pass per sequence and head).
 *   workspace : device memory of kda_chunk_fwd_host_workspace_size() bytes,
 *               16-byte aligned, owned by the caller: device copies of every
 *               input and output, then kda_chunk_fwd's workspace.
 * The prefill runs in rounds of chunks (its segments); the copies follow
 * them: each round's token rows are copied in on a copy stream while earlier
 * rounds compute, and its output rows are copied back on another copy stream
 * once the round's state pass ends.  The call is asynchronous on `stream`:
 * work queued on `stream` afterwards starts only when every copy back has
 * landed.  The two copy streams are made once per device and kept for the
 * life of the process.
 */
KDA_API kda_status_t kda_chunk_fwd_host(const void* q, const void* k, const void* v,
                                        const void* log_alpha, const void* beta,
                                        const float* initial_state, void* out,
                                        kda_dtype_t out_dtype, float* final_state, int B, int T,
                                        int H, int d_k, int d_v, float scale, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream);
KDA_API size_t kda_chunk_fwd_host_workspace_size(int B, int T, int H, int d_k, int d_v,
                                                 kda_dtype_t out_dtype);

/*
 * kda_chunk_bwd -- backward of kda_chunk_fwd, for training: the gradients of
 *   L = <d_out, out> + <d_final_state, final_state>
 * with respect to q, k, v, log_alpha, beta and initial_state.  The pages give
 * no backward algorithm (the studioglobal.ai page, section "Grosse
 * Kapazitaet...", names training at 8k and then 64k contexts); this is the
 * reverse-mode derivative of the token recurrence that kda_chunk_fwd
 * evaluates, S'_t = Diag(alpha_t) S_{t-1}, u_t = beta_t (v_t - S'_t^T k_t),
 * S_t = S'_t + k_t u_t^T, o_t = scale S_t^T q_t.
 *   q, k, v, log_alpha, beta, initial_state, B, T, H, d_k, d_v, scale :
 *                      the forward's arguments, as in kda_chunk_fwd
 *   d_out            : [B, T, H, d_v] fp32, 16-byte aligned
 *   d_final_state    : [B, H, d_k, d_v] fp32, 16-byte aligned, or NULL (zero)
 *   dq, dk, dlog_alpha: [B, T, H, d_k] fp32, 16-byte aligned
 *   dv               : [B, T, H, d_v] fp32, 16-byte aligned
 *   dbeta            : [B, T, H] fp32, 4-byte aligned
 *   d_initial_state  : [B, H, d_k, d_v] fp32, 16-byte aligned, or NULL (not
 *                      written)
 *   workspace        : kda_chunk_bwd_workspace_size(B, T, H, d_k, d_v) bytes,
 *                      16-byte aligned, owned by the caller; it holds the
 *                      forward's records, the state at every 64-token
 *                      boundary, every token's u (fp32, the size of an fp32
 *                      output) and 1 MiB (d = 128) of scratch per sequence
 *                      and head.
 * Every gradient buffer is written in full.  The call runs the forward again
 * (its outputs are not written; where B * H is at most half the SMs it takes
 * the fused launch, which also leaves every token's u) and then one warp per
 * (sequence, head, 4 value columns) over the tokens in reverse, so its time
 * grows with T per sequence and head.
 * Errors are those of kda_chunk_fwd; a NULL gradient buffer other than
 * d_initial_state is KDA_ERR_INVALID_ARG.
 */
KDA_API kda_status_t kda_chunk_bwd(const void* q, const void* k, const void* v,
                                   const void* log_alpha, const void* beta,
                                   const float* initial_state, const float* d_out,
                                   const float* d_final_state, float* dq, float* dk, float* dv,
                                   float* dlog_alpha, float* dbeta, float* d_initial_state, int B,
                                   int T, int H, int d_k, int d_v, float scale, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream);
KDA_API size_t kda_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v);

/* Kernel launches one kda_chunk_fwd call of this shape makes on the current
 * device (the schedule depends on the device's SM count and on
 * KDA_SCHEDULE): 1 for the fused launch, 2 for the plain two-stage
 * schedule, 2 per segment for the overlapped one, more with the segment
 * scan.  -1 on a bad argument or a CUDA error.  A diagnostic for profiling
 * and benchmarks. */
KDA_API int kda_chunk_fwd_launches(int B, int T, int H);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd for callers that are not allowed to
 * allocate device memory at all: for example code whose device memory is
 * budgeted up front by a serving runtime, or code running on a thread that
 * must not call into an allocator.  (The pages have no counterpart; this is
 * an interface convenience of this library.)
 *
 * Same arguments, layouts and results as kda_chunk_fwd, minus the workspace:
 * the intermediate records go to a fixed 64 MiB device array inside the
 * library instead.  Every GPU that loads the library holds that array until
 * the process exits.  Limits and behaviour:
 *   - B * ceil(T / 64) * H must be at most 1008 (one 65 KiB record per chunk
 *     and head); larger problems return KDA_ERR_WORKSPACE before anything
 *     is launched.  Use kda_chunk_fwd with a caller workspace for those.
 *   - All calls share the array.  Calls whose work overlaps on the GPU (two
 *     streams, or two host threads) race on it; serialise them.
 *   - Every call looks up the array's device address on the current
 *     device (a lookup, not an allocation).  The first lookup on a device
 *     may load the library's device code there, so make the first call on
 *     each device before any stream capture.
 */
KDA_API kda_status_t kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                           const void* log_alpha, const void* beta,
                                           const float* initial_state, void* out,
                                           kda_dtype_t out_dtype, float* final_state, int B,
                                           int T, int H, int d_k, int d_v, float scale,
                                           cudaStream_t stream);

/*
 * kda_varlen_fwd -- chunked prefill of N packed sequences of unequal length.
 *   q, k, log_alpha : [T_total, H, d_k] bf16 (a leading batch of 1 is implied)
 *   v               : [T_total, H, d_v] bf16;   beta : [T_total, H] bf16
 *   cu_seqlens      : DEVICE int32 [N + 1], non-decreasing, cu[0] = 0,
 *                     cu[N] = T_total; sequence n owns tokens cu[n]..cu[n+1]-1
 *   max_seqlen      : an upper bound on the longest sequence (sizes the work
 *                     list; a longer sequence flags KDA_ERR_INVALID_ARG in
 *                     the device status word)
 *   initial_state   : [N, H, d_k, d_v] fp32 or NULL;  final_state likewise
 *   out             : [T_total, H, d_v]
 *   workspace       : at least kda_varlen_fwd_workspace_size() bytes
 * Each packed sequence is one request with a fixed-size state of its own
 * (orkas.ai, "Kimi K3 architecture", section "Die Rechnung landet in der
 * Bereitstellungsinfrastruktur": the cache of a request holds per-token
 * pages plus one fixed state), so every sequence starts from its own
 * initial state and ends in its own final state.
 * Chunks start at each sequence's first token; a sequence's last chunk is
 * masked at its end, so no state leaks between sequences.  The chunk list is
 * planned on the device from cu_seqlens (a prefix sum of ceil(len / 64));
 * the call does not synchronise.  The plan clamps every sequence into
 * [0, T_total) and to max_seqlen tokens, so no kernel reads or writes
 * outside the caller's buffers whatever cu_seqlens holds; when it had to
 * clamp (cu[0] != 0, a decreasing offset, an offset past T_total, or a
 * sequence longer than max_seqlen) it flags KDA_ERR_INVALID_ARG in the
 * device status word, and the outputs of the clamped sequences are
 * unspecified.
 */
KDA_API kda_status_t kda_varlen_fwd(const void* q, const void* k, const void* v,
                            const void* log_alpha, const void* beta,
                            const int* cu_seqlens, int N, int T_total,
                            int max_seqlen, const float* initial_state,
                            void* out, kda_dtype_t out_dtype,
                            float* final_state, int H, int d_k, int d_v,
                            float scale, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/* (T_total / 64 + N) * H * 66560 + N * H * 65536 + 256, plus 4 (3 N + 1)
 * bytes rounded up to 1 KiB. */
KDA_API size_t kda_varlen_fwd_workspace_size(int N, int T_total, int H, int d_k, int d_v);

/*
 * kda_decode_step -- one new token for each of N sequences, state updated IN
 * PLACE (the orkas.ai page, section "Die Rechnung landet in der
 * Bereitstellungsinfrastruktur": the state is updated directly and serially).
 *   q, k, log_alpha : [N, H, d_k] bf16;  v : [N, H, d_v] bf16;  beta : [N, H] bf16
 *   state           : [N, H, d_k, d_v] fp32, read and overwritten
 *   out             : [N, H, d_v] in out_dtype
 * d_k = d_v = 128 only.  One read and one write of the state per call.
 */
KDA_API kda_status_t kda_decode_step(const void* q, const void* k, const void* v,
                             const void* log_alpha, const void* beta,
                             float* state, void* out, kda_dtype_t out_dtype,
                             int N, int H, int d_k, int d_v, float scale,
                             cudaStream_t stream);

/*
 * Speculative decoding.  The state is updated in place, so a rejected draft
 * cannot be undone; instead the draft's projected inputs (much smaller than
 * the state) are kept and the state is rebuilt on chip from them (orkas.ai,
 * "Kimi K3 architecture", section "Die Rechnung landet in der
 * Bereitstellungsinfrastruktur").  Each call reads the state once.
 *
 * kda_decode_verify -- outputs of K drafted tokens per sequence, the
 * recurrence applied token after token from `state`, which is only read.
 *   q, k, log_alpha : [N, K, H, d_k] bf16;  v : [N, K, H, d_v] bf16
 *   beta            : [N, K, H] bf16;      state : [N, H, d_k, d_v] fp32
 *   out             : [N, K, H, d_v] in out_dtype; token t of sequence n is
 *                     the output kda_decode_step would give after tokens
 *                     0..t of the draft.
 * kda_decode_commit -- advance each sequence's state, in place, by the first
 * accepted[n] tokens of the same draft inputs (accepted: DEVICE int32 [N],
 * clamped to [0, K]); the state afterwards equals that of accepted[n]
 * kda_decode_step calls.
 * Supported head dims: d_k = d_v = 128.
 */
KDA_API kda_status_t kda_decode_verify(const void* q, const void* k, const void* v,
                                       const void* log_alpha, const void* beta,
                                       const float* state, void* out, kda_dtype_t out_dtype,
                                       int N, int K, int H, int d_k, int d_v, float scale,
                                       cudaStream_t stream);
KDA_API kda_status_t kda_decode_commit(const void* q, const void* k, const void* v,
                                       const void* log_alpha, const void* beta, float* state,
                                       const int* accepted, int N, int K, int H, int d_k,
                                       int d_v, cudaStream_t stream);

/* Static description of a status code (never NULL). */
KDA_API const char* kda_status_string(kda_status_t status);

/*
 * Reads and clears the device status word that kernels set on a decay-bound
 * violation (when checking is on), on a wait that hit its iteration limit,
 * on a packed-sequence plan that had to clamp cu_seqlens, or on a state or
 * corrected value outside the fp16 operand range (KDA_ERR_RANGE).
 * Synchronises `stream`.  Returns KDA_OK when nothing was flagged.
 */
KDA_API kda_status_t kda_last_device_status(cudaStream_t stream);

/* Library version string, e.g. "kda-gb300 1.0 sm_103a". */
KDA_API const char* kda_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H */
