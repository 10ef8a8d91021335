// kda_chunk_fwd on host buffers, with the copies overlapped with the work.
//
// The prefill runs in rounds of chunks (the segments of its overlapped
// schedule; one round for short sequences).  A round's intra-chunk stage and
// state pass read only that round's token rows, and its state pass writes
// only that round's output rows, so the copies can follow the rounds: the
// rows of round k are copied in on one stream while earlier rounds compute,
// the compute stream waits for them before launching round k, and round k's
// output rows are copied out on a second stream once its state pass is done,
// in the other direction of the link while later rounds still copy in.
// The segment scan is not used here (its second walk writes every output at
// the end).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kChunk = 64;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Copy streams of the current device, made once and kept for the process.
struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr;
};
CopyStreams g_copy[64];
std::mutex g_copy_mu;

cudaError_t copy_streams(CopyStreams* cs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_copy_mu);
  CopyStreams& c = g_copy[dev];
  if (!c.in) e = cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking);
  if (e == cudaSuccess && !c.out) e = cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking);
  *cs = c;
  return e;
}

// Device copies of the caller's tensors, in the workspace.
struct Layout {
  size_t tok_in, beta, state, tok_out;  // bytes of one tensor of each kind
  size_t off_q, off_k, off_v, off_la, off_beta, off_s0, off_out, off_fin, off_fwd;
};

Layout layout(int B, int T, int H, int d, bool out_f32) {
  Layout L{};
  const size_t rows = (size_t)B * T * H;
  L.tok_in = rows * d * 2;
  L.beta = rows * 2;
  L.state = (size_t)B * H * d * d * sizeof(float);
  L.tok_out = rows * d * (out_f32 ? 4 : 2);
  size_t o = 0;
  L.off_q = o;  o += align256(L.tok_in);
  L.off_k = o;  o += align256(L.tok_in);
  L.off_v = o;  o += align256(L.tok_in);
  L.off_la = o;  o += align256(L.tok_in);
  L.off_beta = o;  o += align256(L.beta);
  L.off_s0 = o;  o += align256(L.state);
  L.off_out = o;  o += align256(L.tok_out);
  L.off_fin = o;  o += align256(L.state);
  L.off_fwd = o;
  return L;
}

// The per-round copies.  Round k: tokens [64 j_lo, 64 (j_lo + len)) of every
// sequence, i.e. B contiguous row ranges of each token tensor.
struct HostPipe final : RoundHooks {
  const ChunkProblem* host = nullptr;  // host pointers
  uint8_t* dev = nullptr;              // workspace base
  Layout L{};
  CopyStreams cs;
  std::vector<cudaEvent_t> events;  // destroyed by the caller of the schedule
  cudaError_t err = cudaSuccess;

  cudaError_t event(cudaEvent_t* ev) {
    cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e == cudaSuccess) events.push_back(*ev);
    return e;
  }
  // rows [t0, t1) of every sequence of a token tensor with `row_bytes` per token
  cudaError_t copy_rows(void* dst, const void* src, size_t row_bytes, int t0, int t1,
                        cudaMemcpyKind kind, cudaStream_t s) {
    const int B = host->n_seq, T = host->T;
    for (int b = 0; b < B && t1 > t0; ++b) {
      const size_t off = ((size_t)b * T + t0) * row_bytes;
      cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(dst) + off,
                                      static_cast<const uint8_t*>(src) + off,
                                      (size_t)(t1 - t0) * row_bytes, kind, s);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  cudaError_t before_round(int j_lo, int len, cudaStream_t stream) override {
    const int t0 = j_lo * kChunk, t1 = std::min(host->T, (j_lo + len) * kChunk);
    const size_t row_in = (size_t)host->H * host->d * 2, row_beta = (size_t)host->H * 2;
    cudaError_t e = cudaSuccess;
    const struct { size_t off; const void* src; size_t row; } in[] = {
        {L.off_q, host->q, row_in}, {L.off_k, host->k, row_in}, {L.off_v, host->v, row_in},
        {L.off_la, host->log_alpha, row_in}, {L.off_beta, host->beta, row_beta}};
    for (const auto& t : in) {
      if (e == cudaSuccess)
        e = copy_rows(dev + t.off, t.src, t.row, t0, t1, cudaMemcpyHostToDevice, cs.in);
    }
    cudaEvent_t landed = nullptr;
    if (e == cudaSuccess) e = event(&landed);
    if (e == cudaSuccess) e = cudaEventRecord(landed, cs.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, landed, 0);
    return err = e;
  }
  cudaError_t after_round(int j_lo, int len, cudaStream_t stream) override {
    const int t0 = j_lo * kChunk, t1 = std::min(host->T, (j_lo + len) * kChunk);
    const size_t row_out = (size_t)host->H * host->d * (host->out_f32 ? 4 : 2);
    cudaEvent_t done = nullptr;
    cudaError_t e = event(&done);
    if (e == cudaSuccess) e = cudaEventRecord(done, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, done, 0);
    if (e == cudaSuccess)
      e = copy_rows(host->out, dev + L.off_out, row_out, t0, t1, cudaMemcpyDeviceToHost, cs.out);
    return err = e;
  }
};

}  // namespace

size_t chunk_host_workspace_bytes(int B, int T, int H, int d, bool out_f32) {
  return layout(B, T, H, d, out_f32).off_fwd + chunk_workspace_bytes(false, B, T, H);
}

cudaError_t launch_chunk_fwd_host(const ChunkProblem& fwd, void* workspace, cudaStream_t stream) {
  HostPipe pipe;
  pipe.host = &fwd;
  pipe.dev = static_cast<uint8_t*>(workspace);
  pipe.L = layout(fwd.n_seq, fwd.T, fwd.H, fwd.d, fwd.out_f32);
  cudaError_t e = copy_streams(&pipe.cs);
  // the copy streams start after the work already queued on the caller's stream
  cudaEvent_t start = nullptr, end = nullptr;
  if (e == cudaSuccess) e = pipe.event(&start);
  if (e == cudaSuccess) e = cudaEventRecord(start, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe.cs.in, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe.cs.out, start, 0);
  if (e == cudaSuccess && fwd.initial_state) {
    e = cudaMemcpyAsync(pipe.dev + pipe.L.off_s0, fwd.initial_state, pipe.L.state,
                        cudaMemcpyHostToDevice, pipe.cs.in);
    cudaEvent_t s0 = nullptr;
    if (e == cudaSuccess) e = pipe.event(&s0);
    if (e == cudaSuccess) e = cudaEventRecord(s0, pipe.cs.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, s0, 0);
  }
  if (e == cudaSuccess) {
    ChunkProblem p = fwd;
    p.q = pipe.dev + pipe.L.off_q;
    p.k = pipe.dev + pipe.L.off_k;
    p.v = pipe.dev + pipe.L.off_v;
    p.log_alpha = pipe.dev + pipe.L.off_la;
    p.beta = pipe.dev + pipe.L.off_beta;
    p.initial_state = fwd.initial_state ? reinterpret_cast<const float*>(pipe.dev + pipe.L.off_s0)
                                        : nullptr;
    p.out = pipe.dev + pipe.L.off_out;
    p.final_state = fwd.final_state ? reinterpret_cast<float*>(pipe.dev + pipe.L.off_fin) : nullptr;
    p.scan_segs = 0;
    p.hooks = &pipe;
    e = launch_chunk_fwd(p, pipe.dev + pipe.L.off_fwd, stream);
    if (e == cudaSuccess) e = pipe.err;
  }
  if (e == cudaSuccess && fwd.final_state) {  // after the last state pass (or the copy of s0)
    cudaEvent_t done = nullptr;
    e = pipe.event(&done);
    if (e == cudaSuccess) e = cudaEventRecord(done, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe.cs.out, done, 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(fwd.final_state, pipe.dev + pipe.L.off_fin, pipe.L.state,
                          cudaMemcpyDeviceToHost, pipe.cs.out);
  }
  // the caller's stream continues once every copy back has landed
  if (e == cudaSuccess) e = pipe.event(&end);
  if (e == cudaSuccess) e = cudaEventRecord(end, pipe.cs.out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, end, 0);
  for (cudaEvent_t ev : pipe.events) cudaEventDestroy(ev);  // released once complete
  return e;
}

}  // namespace kda
