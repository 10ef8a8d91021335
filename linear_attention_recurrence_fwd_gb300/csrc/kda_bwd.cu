// Backward pass of the KDA layer: the gradients of
//   L = <dO, O> + <dS_T, S_T>
// with respect to q, k, v, log_alpha, beta and the initial state, for the
// recurrence the forward computes (per sequence and head, S is d_k x d_v):
//   S'_t = Diag(alpha_t) S_{t-1},  w_t = v_t - S'_t^T k_t,  u_t = beta_t w_t,
//   S_t  = S'_t + k_t u_t^T,       o_t = scale S_t^T q_t.
// The pages give no backward algorithm (the studioglobal.ai page, section
// "Grosse Kapazitaet...", names training at 8k and then 64k contexts); this
// is reverse-mode differentiation of that recurrence, token by token:
//   G   += scale q_t do_t^T                  (G: gradient of S_t)
//   dq_t = scale S_t do_t,   du = G^T k_t,   dv_t = beta_t du,
//   dbeta_t = du . w_t,      dk_t = G u_t - beta_t S'_t du,
//   dS'  = G - beta_t k_t du^T,  dlog_alpha_t = rowsum(dS' o S'_t),
//   G    = Diag(alpha_t) dS'                  (gradient of S_{t-1}).
//
// Layout of the work: the forward (the chunked tensor-core path) saves the
// state at every chunk boundary; one CTA per (sequence, head) then walks the
// chunks from last to first.  For each chunk it recomputes the 64 token
// states in fp32 from the saved chunk-start state (S'_t to a per-CTA scratch
// in global memory, u_t and w_t to shared memory), then runs the reverse
// recurrence above over the chunk's tokens.  Thread (row c, quarter vg)
// holds G[c][32 vg .. 32 vg + 31] in registers: dot products along a row
// take two shuffles, sums down a column (w and du) a warp reduce-scatter and
// one pass over shared memory.  This is CUDA-core work, serial in tokens per
// (sequence, head): a first, exact formulation, not a tensor-core one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int BW_CH = 64;  // tokens per chunk (the forward's chunk)

struct BwdParams {
  const __nv_bfloat16 *q, *k, *v, *la, *beta;  // [B][T][H][d], beta [B][T][H]
  const float* s0;    // [B][H][d][d] or null (zeros)
  const float* ckpt;  // [B][n_ckpt][H][d][d]: entry m = state after (m + 1) * 64 tokens
  const float* dout;  // [B][T][H][d]
  const float* dfin;  // [B][H][d][d] or null (zeros)
  float *dq, *dk, *dv, *dla, *dbeta, *ds0;
  float* scratch;  // [B * H][64][d][d]
  int T, H, n_ckpt;
  float scale;
};

template <int DIN>
struct BwdShape {
  static constexpr int THREADS = DIN * 4;   // four threads per key row
  static constexpr int NV = DIN / 4;        // value columns per thread
  static constexpr int WARPS = THREADS / 32;
  // shared memory: q, k, log alpha, v (bf16), do (fp32), u, w (fp32), the
  // column-sum partials, one vector, beta
  static constexpr size_t OFF_Q = 0;
  static constexpr size_t OFF_K = OFF_Q + BW_CH * DIN * 2;
  static constexpr size_t OFF_LA = OFF_K + BW_CH * DIN * 2;
  static constexpr size_t OFF_V = OFF_LA + BW_CH * DIN * 2;
  static constexpr size_t OFF_DO = OFF_V + BW_CH * DIN * 2;
  static constexpr size_t OFF_U = OFF_DO + BW_CH * DIN * 4;
  static constexpr size_t OFF_W = OFF_U + BW_CH * DIN * 4;
  static constexpr size_t OFF_RED = OFF_W + BW_CH * DIN * 4;
  static constexpr size_t OFF_VEC = OFF_RED + WARPS * DIN * 4;
  static constexpr size_t OFF_BETA = OFF_VEC + DIN * 4;
  static constexpr size_t SMEM = OFF_BETA + BW_CH * 4;
};

__device__ __forceinline__ float bfv(const __nv_bfloat16* p, int i) {
  return __bfloat162float(p[i]);
}

// Sum over the four threads of a key row.
__device__ __forceinline__ float row_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// Column sums of x (this thread's NV columns of row c) over all DIN rows,
// left in red[] as per-warp partials: a reduce-scatter over the warp's eight
// rows (lane bits 2..4) keeps NV / 8 column sums per lane, which it writes
// to red[warp][column].  The caller synchronises and adds the WARPS
// partials of each column.
template <int NV>
__device__ __forceinline__ void column_partials(float (&x)[NV], float* red, int warp, int lane,
                                                int vg, int din) {
#pragma unroll
  for (int step = 0; step < 3; ++step) {
    const int bit = 16 >> step;          // lane bit 4, 3, 2
    const int half = NV >> (step + 1);   // values kept after this step
    const bool up = (lane & bit) != 0;   // keep the upper half of the current range
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? x[i] : x[i + half];
      float keep = up ? x[i + half] : x[i];
      keep += __shfl_xor_sync(0xffffffffu, send, bit);
      x[i] = keep;
    }
  }
  // kept range: NV / 8 columns starting at NV/2 b4 + NV/4 b3 + NV/8 b2
  const int base = ((lane >> 4) & 1) * (NV / 2) + ((lane >> 3) & 1) * (NV / 4) +
                   ((lane >> 2) & 1) * (NV / 8);
#pragma unroll
  for (int i = 0; i < NV / 8; ++i) red[warp * din + NV * vg + base + i] = x[i];
}

template <int DIN>
__global__ void __launch_bounds__(BwdShape<DIN>::THREADS, 1) kda_bwd_kernel(BwdParams p) {
  using S = BwdShape<DIN>;
  constexpr int NV = S::NV;
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* sq = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_Q);
  __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_K);
  __nv_bfloat16* sla = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_LA);
  __nv_bfloat16* sv = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_V);
  float* sdo = reinterpret_cast<float*>(smem + S::OFF_DO);
  float* su = reinterpret_cast<float*>(smem + S::OFF_U);
  float* sw = reinterpret_cast<float*>(smem + S::OFF_W);
  float* red = reinterpret_cast<float*>(smem + S::OFF_RED);
  float* svec = reinterpret_cast<float*>(smem + S::OFF_VEC);
  float* sbeta = reinterpret_cast<float*>(smem + S::OFF_BETA);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid >> 2, vg = tid & 3, v0 = NV * vg;  // key row, first value column
  const int h = blockIdx.x, n = blockIdx.y, H = p.H, T = p.T;
  const size_t dd = (size_t)DIN * DIN;
  const size_t plane = ((size_t)n * H + h) * dd;  // this (sequence, head) in [B][H][d][d]
  float* scratch = p.scratch + ((size_t)n * H + h) * BW_CH * dd;

  float g[NV];  // G[c][v0 ..]: the gradient of the state after the current token
#pragma unroll
  for (int j = 0; j < NV; ++j) g[j] = p.dfin ? p.dfin[plane + (size_t)c * DIN + v0 + j] : 0.f;

  const int nch = (T + BW_CH - 1) / BW_CH;
  for (int ch = nch - 1; ch >= 0; --ch) {
    const int t0 = ch * BW_CH, L = min(BW_CH, T - t0);
    // ---- stage the chunk's token rows
    __syncthreads();  // the previous chunk is done with shared memory
    for (int e = tid; e < BW_CH * DIN / 8; e += S::THREADS) {  // 8 bf16 (16 bytes) at a time
      const int i = e / (DIN / 8), c8 = (e % (DIN / 8)) * 8;
      uint4 zq = make_uint4(0, 0, 0, 0), zk = zq, zl = zq, zv = zq;
      if (i < L) {
        const size_t off = (((size_t)n * T + t0 + i) * H + h) * DIN + c8;
        zq = *reinterpret_cast<const uint4*>(p.q + off);
        zk = *reinterpret_cast<const uint4*>(p.k + off);
        zl = *reinterpret_cast<const uint4*>(p.la + off);
        zv = *reinterpret_cast<const uint4*>(p.v + off);
      }
      *reinterpret_cast<uint4*>(sq + i * DIN + c8) = zq;
      *reinterpret_cast<uint4*>(sk + i * DIN + c8) = zk;
      *reinterpret_cast<uint4*>(sla + i * DIN + c8) = zl;
      *reinterpret_cast<uint4*>(sv + i * DIN + c8) = zv;
    }
    for (int e = tid; e < BW_CH * DIN / 4; e += S::THREADS) {  // 4 floats at a time
      const int i = e / (DIN / 4), c4 = (e % (DIN / 4)) * 4;
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < L) z = *reinterpret_cast<const float4*>(p.dout + (((size_t)n * T + t0 + i) * H + h) * DIN + c4);
      *reinterpret_cast<float4*>(sdo + i * DIN + c4) = z;
    }
    if (tid < BW_CH) sbeta[tid] = tid < L ? bfv(p.beta, (int)(((size_t)n * T + t0 + tid) * H + h)) : 0.f;
    __syncthreads();

    // ---- forward over the chunk from its saved starting state
    float s[NV];
    {
      const float* src = ch == 0 ? (p.s0 ? p.s0 + plane : nullptr)
                                 : p.ckpt + (((size_t)n * p.n_ckpt + (ch - 1)) * H + h) * dd;
#pragma unroll
      for (int j = 0; j < NV; ++j) s[j] = src ? src[(size_t)c * DIN + v0 + j] : 0.f;
    }
    for (int i = 0; i < L; ++i) {
      const float a = __expf(__bfloat162float(sla[i * DIN + c]));
      const float kc = __bfloat162float(sk[i * DIN + c]);
      float x[NV];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        s[j] *= a;  // S'_t
        x[j] = s[j] * kc;
      }
      float* dst = scratch + (size_t)i * dd + (size_t)c * DIN + v0;
#pragma unroll
      for (int j = 0; j < NV; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
      column_partials<NV>(x, red, warp, lane, vg, DIN);
      __syncthreads();
      if (tid < DIN) {  // w = v - S'^T k, u = beta w
        float acc = 0.f;
#pragma unroll
        for (int wp = 0; wp < S::WARPS; ++wp) acc += red[wp * DIN + tid];
        const float w = __bfloat162float(sv[i * DIN + tid]) - acc;
        sw[i * DIN + tid] = w;
        su[i * DIN + tid] = sbeta[i] * w;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < NV; ++j) s[j] += kc * su[i * DIN + v0 + j];  // S_t
    }

    // ---- the reverse recurrence over the chunk's tokens
    for (int i = L - 1; i >= 0; --i) {
      const size_t tok = ((size_t)n * T + t0 + i) * H + h;
      const float qc = __bfloat162float(sq[i * DIN + c]);
      const float kc = __bfloat162float(sk[i * DIN + c]);
      const float a = __expf(__bfloat162float(sla[i * DIN + c]));
      const float b = sbeta[i];
      const float* dov = sdo + i * DIN + v0;
      const float* uv = su + i * DIN + v0;
      float sp[NV];  // S'_t
      {
        const float* src = scratch + (size_t)i * dd + (size_t)c * DIN + v0;
#pragma unroll
        for (int j = 0; j < NV; j += 4) {
          const float4 f = *reinterpret_cast<const float4*>(src + j);
          sp[j] = f.x;
          sp[j + 1] = f.y;
          sp[j + 2] = f.z;
          sp[j + 3] = f.w;
        }
      }
      // G += scale q do^T;  dq = scale S_t do with S_t = S' + k u^T
      float xq = 0.f;
      float x[NV];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const float dov_j = dov[j];
        g[j] += p.scale * qc * dov_j;
        xq += (sp[j] + kc * uv[j]) * dov_j;
        x[j] = g[j] * kc;
      }
      xq = row_sum(xq);
      if (vg == 0) p.dq[tok * DIN + c] = p.scale * xq;
      // du = G^T k
      column_partials<NV>(x, red, warp, lane, vg, DIN);
      __syncthreads();
      if (tid < DIN) {
        float acc = 0.f;
#pragma unroll
        for (int wp = 0; wp < S::WARPS; ++wp) acc += red[wp * DIN + tid];
        svec[tid] = acc;
        p.dv[tok * DIN + tid] = b * acc;
      }
      __syncthreads();
      // dk = G u - beta S' du;  dS' = G - beta k du^T;  dlog_alpha = rowsum(dS' o S')
      float xk = 0.f, xa = 0.f, xb = 0.f;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const float du = svec[v0 + j];
        xk += g[j] * uv[j] - b * sp[j] * du;
        g[j] -= b * kc * du;
        xa += g[j] * sp[j];
        xb += du * sw[i * DIN + v0 + j];  // the same on every row
        g[j] *= a;  // the gradient of S_{t-1}
      }
      xk = row_sum(xk);
      xa = row_sum(xa);
      xb = row_sum(xb);
      if (vg == 0) {
        p.dk[tok * DIN + c] = xk;
        p.dla[tok * DIN + c] = xa;
        if (c == 0) p.dbeta[tok] = xb;  // dbeta = du . w
      }
    }
  }
  if (p.ds0) {
#pragma unroll
    for (int j = 0; j < NV; ++j) p.ds0[plane + (size_t)c * DIN + v0 + j] = g[j];
  }
}

template <int DIN>
cudaError_t launch_bwd_kernel(const BwdParams& bp, int B, int H, cudaStream_t stream) {
  using S = BwdShape<DIN>;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_kernel<DIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::SMEM);
  if (e != cudaSuccess) return e;
  kda_bwd_kernel<DIN><<<dim3((unsigned)H, (unsigned)B), S::THREADS, S::SMEM, stream>>>(bp);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

// Workspace of the backward: the forward's own workspace, the state at every
// chunk boundary, and the per-(sequence, head) scratch of one chunk's states.
size_t chunk_bwd_workspace_bytes(int B, int T, int H, int d) {
  const size_t dd = (size_t)d * d * sizeof(float);
  const size_t n_ckpt = (size_t)(T / BW_CH);
  return align256(chunk_workspace_bytes(false, B, T, H)) + align256((size_t)B * n_ckpt * H * dd) +
         align256((size_t)B * H * BW_CH * dd);
}

cudaError_t launch_chunk_bwd(const ChunkProblem& fwd, const float* d_out, const float* d_final,
                             float* dq, float* dk, float* dv, float* dla, float* dbeta, float* ds0,
                             void* workspace, cudaStream_t stream) {
  const int B = fwd.n_seq, T = fwd.T, H = fwd.H, d = fwd.d;
  const size_t dd = (size_t)d * d * sizeof(float);
  const int n_ckpt = T / BW_CH;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* fwd_ws = ws;
  float* ckpt = reinterpret_cast<float*>(ws + align256(chunk_workspace_bytes(false, B, T, H)));
  float* scratch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ckpt) +
                                            align256((size_t)B * n_ckpt * H * dd));
  // the forward, for the state at every chunk boundary (its outputs are not needed)
  ChunkProblem f = fwd;
  f.out = nullptr;
  f.final_state = nullptr;
  f.ckpt = n_ckpt > 0 ? ckpt : nullptr;
  f.ckpt_every_chunks = 1;
  f.n_ckpt = n_ckpt;
  f.scan_segs = 0;
  cudaError_t e = launch_chunk_fwd(f, fwd_ws, stream);
  if (e != cudaSuccess) return e;
  BwdParams bp{static_cast<const __nv_bfloat16*>(fwd.q), static_cast<const __nv_bfloat16*>(fwd.k),
               static_cast<const __nv_bfloat16*>(fwd.v), static_cast<const __nv_bfloat16*>(fwd.log_alpha),
               static_cast<const __nv_bfloat16*>(fwd.beta), fwd.initial_state, ckpt, d_out, d_final,
               dq, dk, dv, dla, dbeta, ds0, scratch, T, H, n_ckpt, fwd.scale};
  return d == 64 ? launch_bwd_kernel<64>(bp, B, H, stream) : launch_bwd_kernel<128>(bp, B, H, stream);
}

}  // namespace kda
