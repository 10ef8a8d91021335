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
  __shared__ float s_part[2][8][HALF];  // [a|b][row group][column]
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
  __shared__ float s_u[HALF];
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
template <typename OutT>
__global__ void __launch_bounds__(128) decode_tokens_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ log_alpha,
    const __nv_bfloat16* __restrict__ beta, const float* state_in, float* state_out,
    OutT* __restrict__ out, const int* __restrict__ counts, int K, int H, float scale) {
  __shared__ float s_alpha[DK], s_k[DK], s_q[DK];
  __shared__ float s_part[2][8][HALF];
  __shared__ float s_kq[4];
  __shared__ float s_u[HALF];

  const int tid = threadIdx.x;
  const int nh = blockIdx.x >> 1, half = blockIdx.x & 1;
  const int n = nh / H, h = nh - n * H;
  const int steps = counts ? min(max(counts[n], 0), K) : K;
  const int j = tid & 15, g = tid >> 4;
  constexpr int ROW_F4 = DV / 4;
  const size_t s_off = (size_t)nh * DK * DV;
  const float4* Sin = reinterpret_cast<const float4*>(state_in + s_off) + half * (HALF / 4) + j;

  float4 s[ROWS_PER_THREAD];
#pragma unroll
  for (int i = 0; i < ROWS_PER_THREAD; ++i) s[i] = Sin[(size_t)(g * ROWS_PER_THREAD + i) * ROW_F4];

  for (int t = 0; t < steps; ++t) {
    const size_t row = (size_t)(n * K + t) * H + h;  // (n, t, h)
    __syncthreads();  // the previous token's readers of the shared vectors are done
    {
      const float la = __bfloat162float(log_alpha[row * DK + tid]);
      const float kc = __bfloat162float(k[row * DK + tid]);
      const float qc = __bfloat162float(q[row * DK + tid]);
      s_alpha[tid] = expf(la);
      s_k[tid] = kc;
      s_q[tid] = qc;
      float kq = kc * qc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
      if ((tid & 31) == 0) s_kq[tid >> 5] = kq;
    }
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
    if (tid < HALF) {
      float at = 0.f, bt = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        at += s_part[0][r][tid];
        bt += s_part[1][r][tid];
      }
      const int col = half * HALF + tid;
      const float u = __bfloat162float(beta[row]) * (__bfloat162float(v[row * DV + col]) - at);
      s_u[tid] = u;
      if (out) store_out(out + row * DV + col, scale * (bt + u * (s_kq[0] + s_kq[1] + s_kq[2] + s_kq[3])));
    }
    __syncthreads();
    const float4 u = *reinterpret_cast<const float4*>(&s_u[4 * j]);
#pragma unroll
    for (int i = 0; i < ROWS_PER_THREAD; ++i) {
      const float kc = s_k[g * ROWS_PER_THREAD + i];
      s[i].x += kc * u.x; s[i].y += kc * u.y; s[i].z += kc * u.z; s[i].w += kc * u.w;
    }
  }
  if (state_out) {
    float4* Sout = reinterpret_cast<float4*>(state_out + s_off) + half * (HALF / 4) + j;
#pragma unroll
    for (int i = 0; i < ROWS_PER_THREAD; ++i) Sout[(size_t)(g * ROWS_PER_THREAD + i) * ROW_F4] = s[i];
  }
}

}  // namespace

cudaError_t launch_decode_tokens(const void* q, const void* k, const void* v,
                                 const void* log_alpha, const void* beta, const float* state_in,
                                 float* state_out, void* out, bool out_f32, const int* counts,
                                 int N, int K, int H, float scale, cudaStream_t stream) {
  const long long blocks = 2LL * N * H;
  if (blocks == 0 || K == 0) return cudaSuccess;
  const dim3 grid((unsigned)blocks);
  auto bf = [](const void* p) { return static_cast<const __nv_bfloat16*>(p); };
  if (out_f32 || !out)
    decode_tokens_kernel<float><<<grid, 128, 0, stream>>>(
        bf(q), bf(k), bf(v), bf(log_alpha), bf(beta), state_in, state_out,
        static_cast<float*>(out), counts, K, H, scale);
  else
    decode_tokens_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(
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
