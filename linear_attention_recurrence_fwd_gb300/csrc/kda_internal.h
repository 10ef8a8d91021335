// Internal declarations shared by the host API and the kernel translation
// units of libkda.  Not installed; the public interface is include/kda.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime_api.h>

namespace kda {

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

cudaError_t launch_decode_step(const void* q, const void* k, const void* v,
                               const void* log_alpha, const void* beta, float* state, void* out,
                               bool out_f32, int N, int H, float scale, cudaStream_t stream);

// K tokens per (sequence, head) from one read of the state (see kda_decode.cu).
cudaError_t launch_decode_tokens(const void* q, const void* k, const void* v,
                                 const void* log_alpha, const void* beta, const float* state_in,
                                 float* state_out, void* out, bool out_f32, const int* counts,
                                 int N, int K, int H, float scale, cudaStream_t stream);

// Chunked prefill over either B fixed-length sequences (cu_seqlens == null,
// every sequence T tokens, tensors [B,T,H,d]) or N packed sequences
// (cu_seqlens on the device, tensors [T_total,H,d]).
// Called by the prefill's schedule around each of its rounds (chunks
// [j_lo, j_lo + len) of every sequence), on the compute stream: before the
// round's intra-chunk stage is launched, and after its state pass is.
struct RoundHooks {
  virtual cudaError_t before_round(int j_lo, int len, cudaStream_t stream) = 0;
  virtual cudaError_t after_round(int j_lo, int len, cudaStream_t stream) = 0;

 protected:
  ~RoundHooks() = default;
};

struct ChunkProblem {
  const void *q, *k, *v, *log_alpha, *beta;
  const float* initial_state;
  void* out;
  bool out_f32;
  float* final_state;
  const int* cu_seqlens;  // device, or null
  int n_seq;              // B or N
  int T;                  // tokens per sequence (fixed) or max_seqlen (packed)
  int T_total;            // rows of the token-major tensors
  int H, d;
  float scale;
  bool check_decay;
  bool diag_per_pair;  // ablation: diagonal tiles per position pair on CUDA cores
  // state checkpoints (fixed-length only): after every ckpt_every_chunks
  // chunks of a sequence, n_ckpt of them, [n_seq][n_ckpt][H][d][d]
  float* ckpt;
  int ckpt_every_chunks, n_ckpt;
  // segment scan of fixed-length sequences: -1 lets the library choose, 0
  // or 1 asks for none, more asks for that many segments of whole chunks
  int scan_segs;
  // per-round callbacks (fixed lengths without a scan only), or null
  RoundHooks* hooks = nullptr;
  // or null: every token's u = beta (v - S'^T k), fp32, laid out like an fp32
  // output.  Only the fused launch writes it (fixed lengths, no scan, at most
  // half the SMs in chains: chunk_fwd_writes_u); otherwise the call returns
  // cudaErrorNotSupported before any launch.
  float* u_out = nullptr;
};

// Device workspace the chunked prefill needs: per-(chunk, head) records
// (and, for packed sequences, the per-sequence chunk offsets).
size_t chunk_workspace_bytes(bool packed, int n_seq, long long T_or_total, int H);
// The same for B fixed-length sequences cut into segs segments (a scan).
size_t chunk_scan_workspace_bytes(int B, long long T, int H, int segs);
// Whether a fixed-length forward of n_seq x H chains without a scan can
// write u (ChunkProblem::u_out) on the current device.
bool chunk_fwd_writes_u(int n_seq, int H);

cudaError_t launch_chunk_fwd(const ChunkProblem& p, void* workspace, cudaStream_t stream);

// kda_chunk_fwd on host buffers: the inputs are copied in round by round on
// a copy stream while earlier rounds compute, and each round's outputs are
// copied back as soon as its state pass ends.  fwd holds host pointers; the
// device workspace holds device copies of every input and output, then the
// prefill's own workspace.
size_t chunk_host_workspace_bytes(int B, int T, int H, int d, bool out_f32);
cudaError_t launch_chunk_fwd_host(const ChunkProblem& fwd, void* workspace, cudaStream_t stream);

// Backward of the fixed-length prefill described by fwd (its out and
// final_state are ignored): the forward again for the state at every chunk
// boundary, then the reverse recurrence.  Gradients are fp32 in the layouts
// of the inputs; d_final, ds0 may be null.
size_t chunk_bwd_workspace_bytes(int B, int T, int H, int d);
cudaError_t launch_chunk_bwd(const ChunkProblem& fwd, const float* d_out, const float* d_final,
                             float* dq, float* dk, float* dv, float* dla, float* dbeta, float* ds0,
                             void* workspace, cudaStream_t stream);

// Kernel launches one prefill call of this shape makes on the current device.
int chunk_fwd_launches(bool packed, int n_seq, int max_len, int H);

// Same path with the library's fixed device scratch instead of a caller
// workspace (fixed-length problems of at most noalloc_max_records() records).
size_t noalloc_max_records();
cudaError_t launch_chunk_fwd_noalloc(const ChunkProblem& p, cudaStream_t stream);

// Device status word of the chunk kernels (0 = ok, else a kda_status_t).
int read_and_clear_chunk_status(cudaStream_t stream, cudaError_t* err);

}  // namespace kda
