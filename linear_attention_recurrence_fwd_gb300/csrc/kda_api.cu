// C-ABI boundary of libkda: argument validation, status codes and dispatch
// to the kernels.  No allocation, no printing, no exception crosses it.
#include <cstdint>
#include <cstdlib>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

bool check_decay_env() {
  static int cached = -1;
  if (cached < 0) {
    const char* e = std::getenv("KDA_CHECK_DECAY");
    cached = (e && e[0] && e[0] != '0') ? 1 : 0;
  }
  return cached == 1;
}

// Ablation switch, read on every call: KDA_ABLATE_DIAG=1 evaluates the
// diagonal tiles per position pair instead of with the dense products.
bool ablate_diag_env() {
  const char* e = std::getenv("KDA_ABLATE_DIAG");
  return e && e[0] && e[0] != '0';
}

// The intra-chunk stage walks a work list of (sequence, chunk, head) items
// indexed by int; sequences x chunks of the longest x heads must stay below this.
constexpr long long kMaxItems = 1LL << 30;
long long work_items(int n_seq, int max_len, int H) {
  return (long long)n_seq * ((max_len + 63) / 64) * H;
}

kda_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

kda_status_t validate_prefill(const void* q, const void* k, const void* v, const void* la,
                              const void* beta, const float* s0, const void* out,
                              kda_dtype_t out_dtype, const float* s1, int H, int dk, int dv,
                              bool has_tokens) {
  // token tensors may be empty (null) when there are no tokens at all
  if (has_tokens && (!q || !k || !v || !la || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if (H <= 0 || dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARG;
  if (out_dtype != KDA_BF16 && out_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (dk != dv || !(dk == 128 || dk == 64)) return KDA_ERR_UNSUPPORTED;
  // q, k, v, log_alpha are read by TMA (16-byte rule); beta is read per element
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(la) || !aligned2(beta) ||
      !aligned16(out) || (s0 && !aligned16(s0)) || (s1 && !aligned16(s1)))
    return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

}  // namespace

extern "C" {

const char* kda_status_string(kda_status_t s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KDA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_DECAY_BOUND: return "log_alpha outside [-5, 0]";
    case KDA_ERR_TIMEOUT: return "device wait timed out";
    case KDA_ERR_WORKSPACE: return "workspace too small";
    case KDA_ERR_RANGE: return "state-pass operand outside the fp16 range";
  }
  return "unknown status";
}

const char* kda_version(void) { return "kda-gb300 1.0 sm_103a"; }

size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v) {
  (void)d_k;
  (void)d_v;
  if (B <= 0 || T <= 0 || H <= 0) return 0;
  return kda::chunk_workspace_bytes(false, B, T, H);
}
size_t kda_varlen_fwd_workspace_size(int N, int T_total, int H, int d_k, int d_v) {
  (void)d_k;
  (void)d_v;
  if (N <= 0 || T_total <= 0 || H <= 0) return 0;
  return kda::chunk_workspace_bytes(true, N, T_total, H);
}

kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v, const void* log_alpha,
                           const void* beta, const float* initial_state, void* out,
                           kda_dtype_t out_dtype, float* final_state, int B, int T, int H,
                           int d_k, int d_v, float scale, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || T < 0) return KDA_ERR_INVALID_ARG;
  kda_status_t st = validate_prefill(q, k, v, log_alpha, beta, initial_state, out, out_dtype,
                                     final_state, H, d_k, d_v, (long long)B * T > 0);
  if (st != KDA_OK) return st;
  if ((long long)B * T > 0x7fffffffLL || work_items(B, T, H) > kMaxItems) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  const size_t need = kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v);
  if (need && (!workspace || workspace_bytes < need)) return KDA_ERR_WORKSPACE;
  if (need && !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
  kda::ChunkProblem p{q, k, v, log_alpha, beta, initial_state, out, out_dtype == KDA_F32,
                      final_state, nullptr, B, T, B * T, H, d_k, scale, check_decay_env(),
                      ablate_diag_env()};
  p.scan_segs = -1;  // the library decides whether a segment scan pays
  return from_cuda(kda::launch_chunk_fwd(p, workspace, stream));
}

size_t kda_chunk_fwd_segments_workspace_size(int B, int T, int H, int d_k, int d_v,
                                             int n_segments) {
  (void)d_k;
  (void)d_v;
  if (B <= 0 || T <= 0 || H <= 0 || n_segments < 1) return 0;
  return kda::chunk_scan_workspace_bytes(B, T, H, n_segments);
}

kda_status_t kda_chunk_fwd_segments(const void* q, const void* k, const void* v,
                                    const void* log_alpha, const void* beta,
                                    const float* initial_state, void* out, kda_dtype_t out_dtype,
                                    float* final_state, int B, int T, int H, int d_k, int d_v,
                                    float scale, int n_segments, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || T < 0 || n_segments < 1) return KDA_ERR_INVALID_ARG;
  kda_status_t st = validate_prefill(q, k, v, log_alpha, beta, initial_state, out, out_dtype,
                                     final_state, H, d_k, d_v, (long long)B * T > 0);
  if (st != KDA_OK) return st;
  if ((long long)B * T > 0x7fffffffLL || work_items(B, T, H) > kMaxItems) return KDA_ERR_UNSUPPORTED;
  if ((long long)B * n_segments > (1 << 20)) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  const size_t need = kda_chunk_fwd_segments_workspace_size(B, T, H, d_k, d_v, n_segments);
  if (need && (!workspace || workspace_bytes < need)) return KDA_ERR_WORKSPACE;
  if (need && !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
  kda::ChunkProblem p{q, k, v, log_alpha, beta, initial_state, out, out_dtype == KDA_F32,
                      final_state, nullptr, B, T, B * T, H, d_k, scale, check_decay_env(),
                      ablate_diag_env()};
  p.scan_segs = n_segments;
  return from_cuda(kda::launch_chunk_fwd(p, workspace, stream));
}

kda_status_t kda_chunk_fwd_checkpointed(const void* q, const void* k, const void* v,
                                        const void* log_alpha, const void* beta,
                                        const float* initial_state, void* out,
                                        kda_dtype_t out_dtype, float* final_state, int B, int T,
                                        int H, int d_k, int d_v, float scale, float* checkpoints,
                                        int checkpoint_every, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || T < 0 || checkpoint_every <= 0 || checkpoint_every % 64) return KDA_ERR_INVALID_ARG;
  const int n_ckpt = T / checkpoint_every;
  if (n_ckpt > 0 && !checkpoints) return KDA_ERR_INVALID_ARG;
  if (n_ckpt > 0 && !aligned16(checkpoints)) return KDA_ERR_ALIGNMENT;
  kda_status_t st = validate_prefill(q, k, v, log_alpha, beta, initial_state, out, out_dtype,
                                     final_state, H, d_k, d_v, (long long)B * T > 0);
  if (st != KDA_OK) return st;
  if ((long long)B * T > 0x7fffffffLL || work_items(B, T, H) > kMaxItems) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  const size_t need = kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v);
  if (need && (!workspace || workspace_bytes < need)) return KDA_ERR_WORKSPACE;
  if (need && !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
  kda::ChunkProblem p{q, k, v, log_alpha, beta, initial_state, out, out_dtype == KDA_F32,
                      final_state, nullptr, B, T, B * T, H, d_k, scale, check_decay_env(),
                      ablate_diag_env(), n_ckpt > 0 ? checkpoints : nullptr,
                      checkpoint_every / 64, n_ckpt};
  return from_cuda(kda::launch_chunk_fwd(p, workspace, stream));
}

size_t kda_chunk_fwd_host_workspace_size(int B, int T, int H, int d_k, int d_v,
                                         kda_dtype_t out_dtype) {
  if (B <= 0 || T < 0 || H <= 0 || d_k != d_v || !(d_k == 128 || d_k == 64)) return 0;
  if (out_dtype != KDA_BF16 && out_dtype != KDA_F32) return 0;
  return kda::chunk_host_workspace_bytes(B, T, H, d_k, out_dtype == KDA_F32);
}

kda_status_t kda_chunk_fwd_host(const void* q, const void* k, const void* v, const void* log_alpha,
                                const void* beta, const float* initial_state, void* out,
                                kda_dtype_t out_dtype, float* final_state, int B, int T, int H,
                                int d_k, int d_v, float scale, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || T < 0) return KDA_ERR_INVALID_ARG;
  const bool has_tokens = (long long)B * T > 0;
  if (has_tokens && (!q || !k || !v || !log_alpha || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if (H <= 0 || d_k <= 0 || d_v <= 0) return KDA_ERR_INVALID_ARG;
  if (out_dtype != KDA_BF16 && out_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (d_k != d_v || !(d_k == 128 || d_k == 64)) return KDA_ERR_UNSUPPORTED;
  if ((long long)B * T > 0x7fffffffLL || work_items(B, T, H) > kMaxItems) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  const size_t need = kda_chunk_fwd_host_workspace_size(B, T, H, d_k, d_v, out_dtype);
  if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KDA_ERR_ALIGNMENT;
  kda::ChunkProblem p{q, k, v, log_alpha, beta, initial_state, out, out_dtype == KDA_F32,
                      final_state, nullptr, B, T, B * T, H, d_k, scale, check_decay_env(), false};
  return from_cuda(kda::launch_chunk_fwd_host(p, workspace, stream));
}

size_t kda_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v) {
  if (B <= 0 || T <= 0 || H <= 0 || d_k != d_v || !(d_k == 128 || d_k == 64)) return 0;
  return kda::chunk_bwd_workspace_bytes(B, T, H, d_k);
}

kda_status_t kda_chunk_bwd(const void* q, const void* k, const void* v, const void* log_alpha,
                           const void* beta, const float* initial_state, const float* d_out,
                           const float* d_final_state, float* dq, float* dk, float* dv,
                           float* dlog_alpha, float* dbeta, float* d_initial_state, int B, int T,
                           int H, int d_k, int d_v, float scale, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || T < 0) return KDA_ERR_INVALID_ARG;
  const bool has_tokens = (long long)B * T > 0;
  // d_out takes the output's place in the forward's checks (fp32, 16-byte aligned)
  kda_status_t st = validate_prefill(q, k, v, log_alpha, beta, initial_state, d_out, KDA_F32,
                                     d_final_state, H, d_k, d_v, has_tokens);
  if (st != KDA_OK) return st;
  if (has_tokens && (!dq || !dk || !dv || !dlog_alpha || !dbeta)) return KDA_ERR_INVALID_ARG;
  if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dlog_alpha) ||
      (reinterpret_cast<uintptr_t>(dbeta) & 3u) || (d_initial_state && !aligned16(d_initial_state)))
    return KDA_ERR_ALIGNMENT;
  if ((long long)B * T > 0x7fffffffLL || work_items(B, T, H) > kMaxItems) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  if (T == 0) {  // no tokens: the initial state's gradient is the final state's
    if (!d_initial_state) return KDA_OK;
    const size_t bytes = (size_t)B * H * d_k * d_v * sizeof(float);
    return from_cuda(d_final_state ? cudaMemcpyAsync(d_initial_state, d_final_state, bytes,
                                                     cudaMemcpyDeviceToDevice, stream)
                                   : cudaMemsetAsync(d_initial_state, 0, bytes, stream));
  }
  const size_t need = kda_chunk_bwd_workspace_size(B, T, H, d_k, d_v);
  if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KDA_ERR_ALIGNMENT;
  kda::ChunkProblem p{q, k, v, log_alpha, beta, initial_state, nullptr, true,
                      nullptr, nullptr, B, T, B * T, H, d_k, scale, check_decay_env(), false};
  return from_cuda(kda::launch_chunk_bwd(p, d_out, d_final_state, dq, dk, dv, dlog_alpha, dbeta,
                                         d_initial_state, workspace, stream));
}

kda_status_t kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                   const void* log_alpha, const void* beta,
                                   const float* initial_state, void* out, kda_dtype_t out_dtype,
                                   float* final_state, int B, int T, int H, int d_k, int d_v,
                                   float scale, cudaStream_t stream) {
  if (B < 0 || T < 0) return KDA_ERR_INVALID_ARG;
  kda_status_t st = validate_prefill(q, k, v, log_alpha, beta, initial_state, out, out_dtype,
                                     final_state, H, d_k, d_v, (long long)B * T > 0);
  if (st != KDA_OK) return st;
  if ((long long)B * T > 0x7fffffffLL || work_items(B, T, H) > kMaxItems) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  const long long records = (long long)B * ((T + 63) / 64) * H;
  if (records > (long long)kda::noalloc_max_records()) return KDA_ERR_WORKSPACE;
  kda::ChunkProblem p{q, k, v, log_alpha, beta, initial_state, out, out_dtype == KDA_F32,
                      final_state, nullptr, B, T, B * T, H, d_k, scale, check_decay_env(),
                      ablate_diag_env()};
  return from_cuda(kda::launch_chunk_fwd_noalloc(p, stream));
}

kda_status_t kda_varlen_fwd(const void* q, const void* k, const void* v, const void* log_alpha,
                            const void* beta, const int* cu_seqlens, int N, int T_total,
                            int max_seqlen, const float* initial_state, void* out,
                            kda_dtype_t out_dtype, float* final_state, int H, int d_k, int d_v,
                            float scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  if (!cu_seqlens || N < 0 || T_total < 0 || max_seqlen < 0) return KDA_ERR_INVALID_ARG;
  if (N > 0 && max_seqlen == 0 && T_total > 0) return KDA_ERR_INVALID_ARG;
  if (!aligned16(cu_seqlens)) return KDA_ERR_ALIGNMENT;
  kda_status_t st = validate_prefill(q, k, v, log_alpha, beta, initial_state, out, out_dtype,
                                     final_state, H, d_k, d_v, T_total > 0);
  if (st != KDA_OK) return st;
  if (work_items(N, max_seqlen, H) > kMaxItems) return KDA_ERR_UNSUPPORTED;
  if (N == 0) return KDA_OK;
  const size_t need = kda_varlen_fwd_workspace_size(N, T_total, H, d_k, d_v);
  if (need && (!workspace || workspace_bytes < need)) return KDA_ERR_WORKSPACE;
  if (need && !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
  kda::ChunkProblem p{q, k, v, log_alpha, beta, initial_state, out, out_dtype == KDA_F32,
                      final_state, cu_seqlens, N, max_seqlen, T_total, H, d_k, scale,
                      check_decay_env(), ablate_diag_env()};
  return from_cuda(kda::launch_chunk_fwd(p, workspace, stream));
}

kda_status_t kda_decode_step(const void* q, const void* k, const void* v, const void* log_alpha,
                             const void* beta, float* state, void* out, kda_dtype_t out_dtype,
                             int N, int H, int d_k, int d_v, float scale, cudaStream_t stream) {
  if (N < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  if (N > 0 && (!q || !k || !v || !log_alpha || !beta || !state || !out))
    return KDA_ERR_INVALID_ARG;
  if (out_dtype != KDA_BF16 && out_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (d_k != 128 || d_v != 128) return KDA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned2(beta) || !aligned16(state) || !aligned16(out))
    return KDA_ERR_ALIGNMENT;
  if ((long long)N * H > 0x3fffffffLL) return KDA_ERR_UNSUPPORTED;
  if (N == 0) return KDA_OK;
  return from_cuda(kda::launch_decode_step(q, k, v, log_alpha, beta, state, out,
                                           out_dtype == KDA_F32, N, H, scale, stream));
}

int kda_chunk_fwd_launches(int B, int T, int H) {
  if (B < 0 || T < 0 || H <= 0) return -1;
  return kda::chunk_fwd_launches(false, B, T, H);
}

namespace {
kda_status_t validate_multi(const void* q, const void* k, const void* v, const void* log_alpha,
                            const void* beta, const void* state, int N, int K, int H, int d_k,
                            int d_v) {
  if (N < 0 || K < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  if ((long long)N * K > 0 && (!q || !k || !v || !log_alpha || !beta || !state))
    return KDA_ERR_INVALID_ARG;
  if (d_k != 128 || d_v != 128) return KDA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned2(beta) || !aligned16(state))
    return KDA_ERR_ALIGNMENT;
  if ((long long)N * H > 0x3fffffffLL || (long long)N * K * H > 0x7fffffffLL)
    return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}
}  // namespace

kda_status_t kda_decode_verify(const void* q, const void* k, const void* v, const void* log_alpha,
                               const void* beta, const float* state, void* out,
                               kda_dtype_t out_dtype, int N, int K, int H, int d_k, int d_v,
                               float scale, cudaStream_t stream) {
  kda_status_t st = validate_multi(q, k, v, log_alpha, beta, state, N, K, H, d_k, d_v);
  if (st != KDA_OK) return st;
  if (out_dtype != KDA_BF16 && out_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if ((long long)N * K > 0 && (!out || !aligned16(out))) return out ? KDA_ERR_ALIGNMENT : KDA_ERR_INVALID_ARG;
  if ((long long)N * K == 0) return KDA_OK;
  return from_cuda(kda::launch_decode_tokens(q, k, v, log_alpha, beta, state, nullptr, out,
                                             out_dtype == KDA_F32, nullptr, N, K, H, scale,
                                             stream));
}

kda_status_t kda_decode_commit(const void* q, const void* k, const void* v, const void* log_alpha,
                               const void* beta, float* state, const int* accepted, int N, int K,
                               int H, int d_k, int d_v, cudaStream_t stream) {
  kda_status_t st = validate_multi(q, k, v, log_alpha, beta, state, N, K, H, d_k, d_v);
  if (st != KDA_OK) return st;
  if (N > 0 && !accepted) return KDA_ERR_INVALID_ARG;
  if ((long long)N * K == 0) return KDA_OK;
  return from_cuda(kda::launch_decode_tokens(q, k, v, log_alpha, beta, state, state, nullptr,
                                             true, accepted, N, K, H, 1.f, stream));
}

kda_status_t kda_last_device_status(cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  const int s = kda::read_and_clear_chunk_status(stream, &e);
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  return static_cast<kda_status_t>(s);
}

}  // extern "C"
