// KDA decode step: one new token per (sequence, head), fp32 state updated
// in place.  For each (n, h):
//
//     S'  = Diag(exp(log_alpha)) S          (row c of the d_k x d_v state scaled)
//     a   = S'^T k,   b = S'^T q,   kq = k . q
//     u   = beta (v - a)
//     S   = S' + k u^T                      (written back in place)
//     o   = scale (S^T q) = scale (b + u kq)
//
// o is formed from the same pass over S' that forms a, so the state is read
// once and written once: the kernel is bound by HBM bandwidth (128 KiB of
// state traffic per (n, h) against 1.3 KiB of activations).
//
// Launch: one CTA of 128 threads per (n, h, half of d_v).  Thread t owns
// value columns [4 j, 4 j + 4) of the half (j = t % 16) and key rows
// [16 g, 16 g + 16) (g = t / 16), i.e. 16 float4 registers; a warp covers
// two 256-byte row segments per load, so every access is a coalesced
// 128-bit load or store.  The page's in-place, serial state update is the
// one described on orkas.ai, "Kimi K3 architecture", section "Die Rechnung
// landet in der Bereitstellungsinfrastruktur".
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int DK = 128, DV = 128, HALF = 64;
constexpr int ROWS_PER_THREAD = 16;

template <typename OutT>
__global__ void __launch_bounds__(128) decode_step_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ log_alpha,
    const __nv_bfloat16* __restrict__ beta, float* __restrict__ state, OutT* __restrict__ out,
    float scale) {
  __shared__ float s_alpha[DK], s_k[DK], s_q[DK];
  // float4 accesses below: the arrays read or written as float4 are 16-byte aligned
  __shared__ __align__(16) float s_part[2][8][HALF];  // [a|b][row group][column]
  __shared__ float s_kq[4];

  const int tid = threadIdx.x;
  const int nh = blockIdx.x >> 1;     // flattened (n, h)
  const int half = blockIdx.x & 1;    // which 64 value columns
  const size_t vec = (size_t)nh * DK;  // q/k/log_alpha row of this (n, h)

  // activations: 128 key channels, one per thread
  {
    const float la = __bfloat162float(log_alpha[vec + tid]);
    const float kc = __bfloat162float(k[vec + tid]);
    const float qc = __bfloat162float(q[vec + tid]);
    s_alpha[tid] = expf(la);
    s_k[tid] = kc;
    s_q[tid] = qc;
    float kq = kc * qc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
    if ((tid & 31) == 0) s_kq[tid >> 5] = kq;
  }

  const int j = tid & 15;   // float4 column group within the half
  const int g = tid >> 4;   // row group
  float4* S = reinterpret_cast<float4*>(state + (size_t)nh * DK * DV) + half * (HALF / 4) + j;
  constexpr int ROW_F4 = DV / 4;

  float4 s[ROWS_PER_THREAD];
#pragma unroll
  for (int i = 0; i < ROWS_PER_THREAD; ++i) s[i] = S[(size_t)(g * ROWS_PER_THREAD + i) * ROW_F4];
  __syncthreads();

  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
#pragma unroll
  for (int i = 0; i < ROWS_PER_THREAD; ++i) {
    const int c = g * ROWS_PER_THREAD + i;
    const float al = s_alpha[c], kc = s_k[c], qc = s_q[c];
    s[i].x *= al; s[i].y *= al; s[i].z *= al; s[i].w *= al;
    a.x += s[i].x * kc; a.y += s[i].y * kc; a.z += s[i].z * kc; a.w += s[i].w * kc;
    b.x += s[i].x * qc; b.y += s[i].y * qc; b.z += s[i].z * qc; b.w += s[i].w * qc;
  }
  *reinterpret_cast<float4*>(&s_part[0][g][4 * j]) = a;
  *reinterpret_cast<float4*>(&s_part[1][g][4 * j]) = b;
  __syncthreads();

  // 64 columns: finish the reductions over the 8 row groups
  __shared__ __align__(16) float s_u[HALF];
  if (tid < HALF) {
    float at = 0.f, bt = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      at += s_part[0][r][tid];
      bt += s_part[1][r][tid];
    }
    const int col = half * HALF + tid;
    const float bb = __bfloat162float(beta[nh]);
    const float u = bb * (__bfloat162float(v[(size_t)nh * DV + col]) - at);
    s_u[tid] = u;
    const float kq = s_kq[0] + s_kq[1] + s_kq[2] + s_kq[3];
    const float o = scale * (bt + u * kq);
    store_out(out + (size_t)nh * DV + col, o);
  }
  __syncthreads();

  const float4 u = *reinterpret_cast<const float4*>(&s_u[4 * j]);
#pragma unroll
  for (int i = 0; i < ROWS_PER_THREAD; ++i) {
    const float kc = s_k[g * ROWS_PER_THREAD + i];
    float4 w = s[i];
    w.x += kc * u.x; w.y += kc * u.y; w.z += kc * u.z; w.w += kc * u.w;
    S[(size_t)(g * ROWS_PER_THREAD + i) * ROW_F4] = w;
  }
}

// Several tokens per (sequence, head) from one read of the state: the
// speculative-decoding pair.  Token t of sequence n is row (n K + t) of the
// [N, K, H, d] activations.  steps = counts ? clamp(counts[n], 0, K) : K
// tokens are applied to the state held in registers, one after another
// exactly as in decode_step_kernel; o is written for each when out is given,
// and the state after the last applied token is written when state_out is
// given.  Verify: counts = null, state_out = null (the state is only read).
// Commit: counts = accepted, state_out = state, out = null.
// Several tokens per (sequence, head) in order.  The state stays in registers
// across the tokens, so it is read once and written once (or not at all, for
// verification) however many tokens there are.  Each CTA owns d_v / SPLIT
// value columns: thread t holds columns [4 j, 4 j + 4) of them (j = t % TJ)
// for rows [RPT g, RPT g + RPT) (g = t / TJ).  Measured at 256 sequences x
// 32 heads x 4 tokens, halves beat quarters and eighths of d_v: each token's
// barriers and column sums cost the same per CTA whatever its width, so
// narrower CTAs only add CTAs.
template <typename OutT, int SPLIT>
__global__ void __launch_bounds__(128) decode_tokens_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ log_alpha,
    const __nv_bfloat16* __restrict__ beta, const float* state_in, float* state_out,
    OutT* __restrict__ out, const int* __restrict__ counts, int K, int H, float scale) {
  constexpr int COLS = DV / SPLIT;  // value columns of this CTA
  constexpr int TJ = COLS / 4;      // threads across a row (one float4 each)
  constexpr int G = 128 / TJ;       // row groups
  constexpr int RPT = DK / G;       // rows per thread
  // The tokens' activations are staged KT at a time, all loads issued
  // together, so a pass pays one global-memory latency rather than one per
  // token.  Two at a time keeps the kernel at 124 registers, four CTAs per
  // SM; eight took 158 (three CTAs) and verify 7 % longer.
  constexpr int KT = 2;
  __shared__ float s_alpha[KT][DK], s_k[KT][DK], s_q[KT][DK];
  __shared__ float s_v[KT][COLS], s_beta[KT], s_kq[KT][4];
  // read and written as float4: 16-byte aligned whatever precedes them
  __shared__ __align__(16) float s_part[2][G][COLS];
  __shared__ __align__(16) float s_u[COLS];

  const int tid = threadIdx.x;
  const int nh = blockIdx.x / SPLIT, part = blockIdx.x % SPLIT;
  const int n = nh / H, h = nh - n * H;
  const int steps = counts ? min(max(counts[n], 0), K) : K;
  const int j = tid % TJ, g = tid / TJ;
  constexpr int ROW_F4 = DV / 4;
  const size_t s_off = (size_t)nh * DK * DV;
  const float4* Sin = reinterpret_cast<const float4*>(state_in + s_off) + part * TJ + j;

  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = Sin[(size_t)(g * RPT + i) * ROW_F4];

  for (int t0 = 0; t0 < steps; t0 += KT) {
    const int nt = min(KT, steps - t0);
    __syncthreads();  // the previous pass's readers of the staged tokens are done
    __nv_bfloat16 r_la[KT], r_k[KT], r_q[KT], r_v[KT], r_b[KT];
#pragma unroll
    for (int t = 0; t < KT; ++t) {
      if (t < nt) {
        const size_t row = (size_t)(n * K + t0 + t) * H + h;  // (n, t0 + t, h)
        r_la[t] = log_alpha[row * DK + tid];
        r_k[t] = k[row * DK + tid];
        r_q[t] = q[row * DK + tid];
        if (tid < COLS) r_v[t] = v[row * DV + part * COLS + tid];
        if (tid == 0) r_b[t] = beta[row];
      }
    }
#pragma unroll
    for (int t = 0; t < KT; ++t) {
      if (t < nt) {
        const float kc = __bfloat162float(r_k[t]), qc = __bfloat162float(r_q[t]);
        s_alpha[t][tid] = expf(__bfloat162float(r_la[t]));
        s_k[t][tid] = kc;
        s_q[t][tid] = qc;
        if (tid < COLS) s_v[t][tid] = __bfloat162float(r_v[t]);
        if (tid == 0) s_beta[t] = __bfloat162float(r_b[t]);
        float kq = kc * qc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
        if ((tid & 31) == 0) s_kq[t][tid >> 5] = kq;
      }
    }
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int c = g * RPT + i;
        const float al = s_alpha[t][c], kc = s_k[t][c], qc = s_q[t][c];
        s[i].x *= al; s[i].y *= al; s[i].z *= al; s[i].w *= al;
        a.x += s[i].x * kc; a.y += s[i].y * kc; a.z += s[i].z * kc; a.w += s[i].w * kc;
        b.x += s[i].x * qc; b.y += s[i].y * qc; b.z += s[i].z * qc; b.w += s[i].w * qc;
      }
      *reinterpret_cast<float4*>(&s_part[0][g][4 * j]) = a;
      *reinterpret_cast<float4*>(&s_part[1][g][4 * j]) = b;
      __syncthreads();
      if (tid < COLS) {
        float at = 0.f, bt = 0.f;
#pragma unroll
        for (int r = 0; r < G; ++r) {
          at += s_part[0][r][tid];
          bt += s_part[1][r][tid];
        }
        const float u = s_beta[t] * (s_v[t][tid] - at);
        s_u[tid] = u;
        if (out) {
          const size_t row = (size_t)(n * K + t0 + t) * H + h;
          const float kq = s_kq[t][0] + s_kq[t][1] + s_kq[t][2] + s_kq[t][3];
          store_out(out + row * DV + part * COLS + tid, scale * (bt + u * kq));
        }
      }
      __syncthreads();
      const float4 u = *reinterpret_cast<const float4*>(&s_u[4 * j]);
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float kc = s_k[t][g * RPT + i];
        s[i].x += kc * u.x; s[i].y += kc * u.y; s[i].z += kc * u.z; s[i].w += kc * u.w;
      }
      // No barrier here: the next token writes s_part only after every thread
      // has read s_u, and s_u only after the next token's first barrier.
    }
  }
  if (state_out) {
    float4* Sout = reinterpret_cast<float4*>(state_out + s_off) + part * TJ + j;
#pragma unroll
    for (int i = 0; i < RPT; ++i) Sout[(size_t)(g * RPT + i) * ROW_F4] = s[i];
  }
}

}  // namespace

cudaError_t launch_decode_tokens(const void* q, const void* k, const void* v,
                                 const void* log_alpha, const void* beta, const float* state_in,
                                 float* state_out, void* out, bool out_f32, const int* counts,
                                 int N, int K, int H, float scale, cudaStream_t stream) {
  constexpr int SPLIT = 2;
  const long long blocks = (long long)SPLIT * N * H;
  if (blocks == 0 || K == 0) return cudaSuccess;
  const dim3 grid((unsigned)blocks);
  auto bf = [](const void* p) { return static_cast<const __nv_bfloat16*>(p); };
  if (out_f32 || !out)
    decode_tokens_kernel<float, SPLIT><<<grid, 128, 0, stream>>>(
        bf(q), bf(k), bf(v), bf(log_alpha), bf(beta), state_in, state_out,
        static_cast<float*>(out), counts, K, H, scale);
  else
    decode_tokens_kernel<__nv_bfloat16, SPLIT><<<grid, 128, 0, stream>>>(
        bf(q), bf(k), bf(v), bf(log_alpha), bf(beta), state_in, state_out,
        static_cast<__nv_bfloat16*>(out), counts, K, H, scale);
  return cudaGetLastError();
}

cudaError_t launch_decode_step(const void* q, const void* k, const void* v,
                               const void* log_alpha, const void* beta, float* state, void* out,
                               bool out_f32, int N, int H, float scale, cudaStream_t stream) {
  const long long blocks = 2LL * N * H;
  if (blocks == 0) return cudaSuccess;
  const dim3 grid((unsigned)blocks);
  auto bf = [](const void* p) { return static_cast<const __nv_bfloat16*>(p); };
  if (out_f32)
    decode_step_kernel<float><<<grid, 128, 0, stream>>>(
        bf(q), bf(k), bf(v), bf(log_alpha), bf(beta), state, static_cast<float*>(out), scale);
  else
    decode_step_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(
        bf(q), bf(k), bf(v), bf(log_alpha), bf(beta), state, static_cast<__nv_bfloat16*>(out),
        scale);
  return cudaGetLastError();
}

}  // namespace kda
