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
// state at every chunk boundary and, where it can (the fused launch), every
// token's u; one warp per (sequence, head, block of 4 value columns) then
// walks the chunks from last to first.  For each chunk it rebuilds the token
// states in fp32 from the saved chunk-start state: with u given that is a
// local step per token (S'_t = Diag(alpha_t) S_{t-1}, S_t = S'_t + k_t u_t^T,
// w_t = u_t / beta_t), and only without it, or for a token with beta = 0,
// does w take a column sum.  It keeps the state before every 4th token (in a
// per-warp scratch in global memory) and, in the reverse recurrence, rebuilds
// each group of 4 token states in registers from it.  Lane l holds d_k / 32
// consecutive rows of G for the warp's columns in registers: dot products
// along a row stay in the lane, sums down a column (du, and w without u) are
// a shuffle reduction over the warp.  This is CUDA-core work, serial in tokens per
// (sequence, head): an exact token-level formulation, not a tensor-core one.
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
  float* scratch;      // [B * H][d / CW][64 / SUB][d][CW]: per warp, the state before each sub-block
  const float* u_fwd;  // [B][T][H][d]: every token's u from the forward (HAVE_U), or null
  int T, H, n_ckpt;
  float scale;
};

// Work split.  The columns of G evolve independently (each step scales rows
// and adds rank-one terms), so a warp owns a block of CW value columns for
// all d_k key rows, lane l the RL = d_k / 32 consecutive rows RL l, ...:
// a sum down a column (du, and w without u) is then a shuffle reduction over
// the warp's lanes with no barrier.  Only the gradients summed along a row (dq,
// dk, dlog_alpha, dbeta) join the column blocks, by atomic adds into zeroed
// buffers.  A CTA of WPC warps (WPC column blocks of one (sequence, head))
// stages each chunk's token rows once for all its warps; the warps meet only
// at the chunk boundaries.
// Measured on the 8k problem: CW = 4 with 4 warps per CTA 6.8 ms; CW = 2
// 7.9-8.2 ms (more warps, more work per column); CW = 8 8.7-8.9 ms (fewer
// warps, 208-254 registers).
constexpr int CW = 4;   // value columns per warp
constexpr int WPC = 4;  // warps per CTA
// Tokens per sub-block of the reverse pass: the state before each sub-block
// is saved (in the per-warp scratch), and the sub-block's token states are
// rebuilt in registers when the reverse pass reaches it.
constexpr int SUB = 4;

template <int DIN>
struct BwdShape {
  static constexpr int RL = DIN / 32;  // key rows per lane
  static constexpr int THREADS = 32 * WPC;
  static constexpr int COLS = CW * WPC;    // value columns per CTA
  static constexpr int CTAS = DIN / COLS;  // CTAs per (sequence, head)
  static_assert(COLS % 8 == 0 && DIN % COLS == 0, "whole 16-byte rows of v staged per CTA");
  // shared memory: q, k, log alpha (bf16, every channel), the CTA's v
  // columns (bf16), its do, u and w columns (fp32), beta
  static constexpr size_t OFF_Q = 0;
  static constexpr size_t OFF_K = OFF_Q + BW_CH * DIN * 2;
  static constexpr size_t OFF_LA = OFF_K + BW_CH * DIN * 2;
  static constexpr size_t OFF_V = OFF_LA + BW_CH * DIN * 2;
  static constexpr size_t OFF_DO = OFF_V + BW_CH * COLS * 2;
  static constexpr size_t OFF_U = OFF_DO + BW_CH * COLS * 4;
  static constexpr size_t OFF_W = OFF_U + BW_CH * COLS * 4;
  static constexpr size_t OFF_BETA = OFF_W + BW_CH * COLS * 4;
  static constexpr size_t SMEM = OFF_BETA + BW_CH * 4;
};
static_assert(CW == 2 || CW == 4 || CW == 8, "a lane's share of a key row is 8, 16 or 32 bytes");

__device__ __forceinline__ float bfv(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

// The lane's RL consecutive bf16 entries of a staged token row, as floats.
template <int RL>
__device__ __forceinline__ void ld_rows(const __nv_bfloat16* src, float (&x)[RL]) {
  if constexpr (RL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(src);
    x[0] = __uint_as_float(u << 16);
    x[1] = __uint_as_float(u & 0xffff0000u);
  }
}

// Column sums over the warp's lanes, left on every lane: a reduce-scatter
// over the top lane bits (each lane then holds one column's partial), a sum
// over the remaining bits, and one broadcast per column, so that every lane
// ends with the same bits.
__device__ __forceinline__ void warp_sum(float (&y)[CW], int lane) {
  const bool up = (lane & 16) != 0;
  float k;
  if constexpr (CW == 8) {
    const bool up8 = (lane & 8) != 0, up4 = (lane & 4) != 0;
    float k4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      k4[i] = up ? y[i + 4] : y[i];
      k4[i] += __shfl_xor_sync(0xffffffffu, up ? y[i] : y[i + 4], 16);
    }
    float k2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      k2[i] = up8 ? k4[i + 2] : k4[i];
      k2[i] += __shfl_xor_sync(0xffffffffu, up8 ? k4[i] : k4[i + 2], 8);
    }
    k = up4 ? k2[1] : k2[0];  // column 4 (lane bit 4) + 2 (lane bit 3) + (lane bit 2)
    k += __shfl_xor_sync(0xffffffffu, up4 ? k2[0] : k2[1], 4);
  } else if constexpr (CW == 4) {
    const bool up8 = (lane & 8) != 0;
    float k0 = up ? y[2] : y[0], k1 = up ? y[3] : y[1];
    k0 += __shfl_xor_sync(0xffffffffu, up ? y[0] : y[2], 16);
    k1 += __shfl_xor_sync(0xffffffffu, up ? y[1] : y[3], 16);
    k = up8 ? k1 : k0;  // column 2 (lane bit 4) + (lane bit 3)
    k += __shfl_xor_sync(0xffffffffu, up8 ? k0 : k1, 8);
  } else {
    k = up ? y[1] : y[0];  // column (lane bit 4)
    k += __shfl_xor_sync(0xffffffffu, up ? y[0] : y[1], 16);
    k += __shfl_xor_sync(0xffffffffu, k, 8);
  }
  if constexpr (CW != 8) k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
#pragma unroll
  for (int j = 0; j < CW; ++j)
    y[j] = __shfl_sync(0xffffffffu, k,
                       CW == 8   ? (j >> 2) * 16 + ((j >> 1) & 1) * 8 + (j & 1) * 4
                       : CW == 4 ? (j >> 1) * 16 + (j & 1) * 8
                                 : j * 16);
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
// CW consecutive floats (one vector): x = p[0 .. CW), p[0 .. CW) = x
__device__ __forceinline__ void ldw(const float* p, float (&x)[CW]) {
  if constexpr (CW == 8) {
    const float4 f = ld4(p), h = ld4(p + 4);
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
    x[4] = h.x;
    x[5] = h.y;
    x[6] = h.z;
    x[7] = h.w;
  } else if constexpr (CW == 4) {
    const float4 f = ld4(p);
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
  } else {
    const float2 f = *reinterpret_cast<const float2*>(p);
    x[0] = f.x;
    x[1] = f.y;
  }
}
__device__ __forceinline__ void stw(float* p, const float (&x)[CW]) {
  if constexpr (CW == 8) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
  } else if constexpr (CW == 4)
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
}

// Row sums of one token for the lane's RL key rows, added into a gradient.
template <int RL>
__device__ __forceinline__ void add_rows(float* dst, const float (&x)[RL]) {
  if constexpr (RL == 4)
    atomicAdd(reinterpret_cast<float4*>(dst), make_float4(x[0], x[1], x[2], x[3]));
  else
    atomicAdd(reinterpret_cast<float2*>(dst), make_float2(x[0], x[1]));
}

// HAVE_U: the forward left every token's u, so the chunk's token states
// follow from the saved chunk-start state with no column sums (w = u / beta;
// only a token with beta = 0 takes the sum for its w).
template <int DIN, bool HAVE_U>
__global__ void __launch_bounds__(BwdShape<DIN>::THREADS) kda_bwd_kernel(BwdParams p) {
  using S = BwdShape<DIN>;
  constexpr int RL = S::RL, COLS = S::COLS;
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* sq = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_Q);
  __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_K);
  __nv_bfloat16* sla = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_LA);
  __nv_bfloat16* sv = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_V);
  float* sdo = reinterpret_cast<float*>(smem + S::OFF_DO);
  float* su = reinterpret_cast<float*>(smem + S::OFF_U);
  float* sw = reinterpret_cast<float*>(smem + S::OFF_W);
  float* sbeta = reinterpret_cast<float*>(smem + S::OFF_BETA);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, n = blockIdx.y;
  const int cb = COLS * blockIdx.z;  // the CTA's first value column
  const int wc = CW * warp;          // the warp's first column within the CTA's
  const int vb = cb + wc;            // the warp's first value column
  const int r0 = RL * lane;          // the lane's first key row
  const int H = p.H, T = p.T;
  const size_t dd = (size_t)DIN * DIN;
  const size_t plane = ((size_t)n * H + h) * dd;  // this (sequence, head) in [B][H][d][d]
  // the warp's scratch of one chunk: the state before each sub-block, laid
  // out [sub-block][lane][RL rows][CW columns]
  float* scratch = p.scratch + (((size_t)n * H + h) * (DIN / CW) + vb / CW) * (BW_CH / SUB) * DIN * CW +
                   (size_t)lane * RL * CW;

  // x = the lane's rows of columns vb .. vb + CW of a [d][d] plane (zeros for null)
  auto load_state = [&](const float* src, float (&x)[RL][CW]) {
#pragma unroll
    for (int m = 0; m < RL; ++m) {
      if (src) {
        ldw(src + (size_t)(r0 + m) * DIN + vb, x[m]);
      } else {
#pragma unroll
        for (int j = 0; j < CW; ++j) x[m][j] = 0.f;
      }
    }
  };
  auto save_sub = [&](int sb, const float (&x)[RL][CW]) {
    float* dst = scratch + (size_t)sb * DIN * CW;
#pragma unroll
    for (int m = 0; m < RL; ++m)
      stw(dst + m * CW, x[m]);
  };
  auto load_sub = [&](int sb, float (&x)[RL][CW]) {
    const float* src = scratch + (size_t)sb * DIN * CW;
#pragma unroll
    for (int m = 0; m < RL; ++m) {
      ldw(src + m * CW, x[m]);
    }
  };

  float g[RL][CW];  // G for the lane's rows and the warp's columns: the gradient of the state after the current token
  load_state(p.dfin ? p.dfin + plane : nullptr, g);

  const int nch = (T + BW_CH - 1) / BW_CH;
  for (int ch = nch - 1; ch >= 0; --ch) {
    const int t0 = ch * BW_CH, L = min(BW_CH, T - t0);
    // ---- stage the chunk's token rows (the CTA's columns of v, do and u)
    __syncthreads();  // every warp is done with the previous chunk
    for (int e = tid; e < BW_CH * DIN / 8; e += S::THREADS) {  // 8 bf16 (16 bytes) at a time
      const int i = e / (DIN / 8), c8 = (e % (DIN / 8)) * 8;
      uint4 zq = make_uint4(0, 0, 0, 0), zk = zq, zl = zq;
      if (i < L) {
        const size_t off = (((size_t)n * T + t0 + i) * H + h) * DIN + c8;
        zq = *reinterpret_cast<const uint4*>(p.q + off);
        zk = *reinterpret_cast<const uint4*>(p.k + off);
        zl = *reinterpret_cast<const uint4*>(p.la + off);
      }
      *reinterpret_cast<uint4*>(sq + i * DIN + c8) = zq;
      *reinterpret_cast<uint4*>(sk + i * DIN + c8) = zk;
      *reinterpret_cast<uint4*>(sla + i * DIN + c8) = zl;
    }
    for (int e = tid; e < BW_CH * COLS / 8; e += S::THREADS) {
      const int i = e / (COLS / 8), c8 = (e % (COLS / 8)) * 8;
      uint4 z = make_uint4(0, 0, 0, 0);
      if (i < L) z = *reinterpret_cast<const uint4*>(p.v + (((size_t)n * T + t0 + i) * H + h) * DIN + cb + c8);
      *reinterpret_cast<uint4*>(sv + i * COLS + c8) = z;
    }
    for (int e = tid; e < BW_CH * COLS / 4; e += S::THREADS) {
      const int i = e / (COLS / 4), c4 = (e % (COLS / 4)) * 4;
      const size_t off = (((size_t)n * T + t0 + i) * H + h) * DIN + cb + c4;
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f), zu = z;
      if (i < L) {
        z = ld4(p.dout + off);
        if (HAVE_U) zu = ld4(p.u_fwd + off);
      }
      *reinterpret_cast<float4*>(sdo + i * COLS + c4) = z;
      if (HAVE_U) *reinterpret_cast<float4*>(su + i * COLS + c4) = zu;
    }
    if (tid < BW_CH) sbeta[tid] = tid < L ? bfv(p.beta, ((size_t)n * T + t0 + tid) * H + h) : 0.f;
    __syncthreads();

    // ---- forward over the chunk from its saved starting state (each warp alone)
    {
      float s[RL][CW];
      load_state(ch == 0 ? (p.s0 ? p.s0 + plane : nullptr)
                         : p.ckpt + (((size_t)n * p.n_ckpt + (ch - 1)) * H + h) * dd,
                 s);
      for (int i = 0; i < L; ++i) {
        float a[RL], kc[RL];
        ld_rows<RL>(sla + i * DIN + r0, a);
        ld_rows<RL>(sk + i * DIN + r0, kc);
        if ((i & (SUB - 1)) == 0) save_sub(i / SUB, s);  // S_{t-1}: the state before this sub-block
#pragma unroll
        for (int m = 0; m < RL; ++m) {
          a[m] = __expf(a[m]);
#pragma unroll
          for (int j = 0; j < CW; ++j) s[m][j] *= a[m];  // S'_t
        }
        float u[CW];
        const float b = sbeta[i];
        if (!HAVE_U || b == 0.f) {  // (the same on every lane) w = v - S'^T k, u = beta w
          float y[CW];
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            y[j] = 0.f;
#pragma unroll
            for (int m = 0; m < RL; ++m) y[j] += s[m][j] * kc[m];
          }
          warp_sum(y, lane);
          float w[CW];
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            w[j] = __bfloat162float(sv[i * COLS + wc + j]) - y[j];
            u[j] = b * w[j];
          }
          if (lane == 0) {
            stw(sw + i * COLS + wc, w);
            stw(su + i * COLS + wc, u);
          }
        } else {
          ldw(su + i * COLS + wc, u);
        }
#pragma unroll
        for (int m = 0; m < RL; ++m) {
#pragma unroll
          for (int j = 0; j < CW; ++j) s[m][j] += kc[m] * u[j];  // S_t
        }
      }
    }
    if (HAVE_U) {  // w = u / beta where beta != 0 (the warp's columns)
      for (int e = lane; e < L * CW; e += 32) {
        const int i = e / CW, j = e % CW;
        const float b = sbeta[i];
        if (b != 0.f) sw[i * COLS + wc + j] = su[i * COLS + wc + j] / b;
      }
    }
    __syncwarp();

    // ---- the reverse recurrence over the chunk's tokens, SUB at a time: the
    // sub-block's S'_t are rebuilt in registers from the state saved before
    // it (a local step per token: u is known), whose load is issued one
    // sub-block ahead.
    const int nsub = (L + SUB - 1) / SUB;
    float nxt[RL][CW];
    if (nsub > 0) load_sub(nsub - 1, nxt);
    for (int sbk = nsub - 1; sbk >= 0; --sbk) {
      float spq[SUB][RL][CW];
      {
        float st[RL][CW];
#pragma unroll
        for (int m = 0; m < RL; ++m) {
#pragma unroll
          for (int j = 0; j < CW; ++j) st[m][j] = nxt[m][j];
        }
        if (sbk > 0) load_sub(sbk - 1, nxt);
#pragma unroll
        for (int q = 0; q < SUB; ++q) {
          const int i = SUB * sbk + q;
          float a[RL], kc[RL], u[CW];
          if (i < L) {
            ld_rows<RL>(sla + i * DIN + r0, a);
            ld_rows<RL>(sk + i * DIN + r0, kc);
            ldw(su + i * COLS + wc, u);
#pragma unroll
            for (int m = 0; m < RL; ++m) a[m] = __expf(a[m]);
          } else {
#pragma unroll
            for (int m = 0; m < RL; ++m) {
              a[m] = 1.f;
              kc[m] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < CW; ++j) u[j] = 0.f;
          }
#pragma unroll
          for (int m = 0; m < RL; ++m) {
#pragma unroll
            for (int j = 0; j < CW; ++j) {
              st[m][j] *= a[m];
              spq[q][m][j] = st[m][j];
              st[m][j] += kc[m] * u[j];
            }
          }
        }
      }
#pragma unroll
      for (int q = SUB - 1; q >= 0; --q) {
        const int i = SUB * sbk + q;
        if (i >= L) continue;  // (the same on every lane)
        const size_t tok = ((size_t)n * T + t0 + i) * H + h;
        float qc[RL], kc[RL], a[RL];
        ld_rows<RL>(sq + i * DIN + r0, qc);
        ld_rows<RL>(sk + i * DIN + r0, kc);
        ld_rows<RL>(sla + i * DIN + r0, a);
        const float b = sbeta[i];
        float dov[CW], uv[CW], wv[CW];
        ldw(sdo + i * COLS + wc, dov);
        ldw(su + i * COLS + wc, uv);
        ldw(sw + i * COLS + wc, wv);
        // G += scale q do^T, then du = G^T k
        float du[CW];
#pragma unroll
        for (int j = 0; j < CW; ++j) du[j] = 0.f;
#pragma unroll
        for (int m = 0; m < RL; ++m) {
          const float sq_m = p.scale * qc[m];
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            g[m][j] += sq_m * dov[j];
            du[j] += g[m][j] * kc[m];
          }
        }
        warp_sum(du, lane);
        if (lane == 0) {  // dv = beta du, and this block's share of dbeta = du . w
          float dvv[CW], db = 0.f;
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            dvv[j] = b * du[j];
            db += du[j] * wv[j];
          }
          stw(p.dv + tok * DIN + vb, dvv);
          atomicAdd(p.dbeta + tok, db);
        }
        // dq = scale S_t do with S_t = S' + k u^T;  dk = G u - beta S' du;
        // dS' = G - beta k du^T;  dlog_alpha = rowsum(dS' o S')  (this warp's columns)
        float ud = 0.f;  // u . do, the same on every row
#pragma unroll
        for (int j = 0; j < CW; ++j) ud += uv[j] * dov[j];
        float xq[RL], xk[RL], xa[RL];
#pragma unroll
        for (int m = 0; m < RL; ++m) {
          const float* sp = spq[q][m];
          const float am = __expf(a[m]), bk = b * kc[m];
          float aq = 0.f, gu = 0.f, sd = 0.f, aa = 0.f;
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            aq += sp[j] * dov[j];
            gu += g[m][j] * uv[j];
            sd += sp[j] * du[j];
            g[m][j] -= bk * du[j];
            aa += g[m][j] * sp[j];
            g[m][j] *= am;  // the gradient of S_{t-1}
          }
          xq[m] = p.scale * (aq + kc[m] * ud);
          xk[m] = gu - b * sd;
          xa[m] = aa;
        }
        add_rows<RL>(p.dq + tok * DIN + r0, xq);
        add_rows<RL>(p.dk + tok * DIN + r0, xk);
        add_rows<RL>(p.dla + tok * DIN + r0, xa);
      }
    }
  }
  if (p.ds0) {
#pragma unroll
    for (int m = 0; m < RL; ++m)
      stw(p.ds0 + plane + (size_t)(r0 + m) * DIN + vb, g[m]);
  }
}

template <int DIN, bool HAVE_U>
cudaError_t launch_bwd_kernel(const BwdParams& bp, int B, int H, cudaStream_t stream) {
  using S = BwdShape<DIN>;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_kernel<DIN, HAVE_U>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
  if (e != cudaSuccess) return e;
  kda_bwd_kernel<DIN, HAVE_U>
      <<<dim3((unsigned)H, (unsigned)B, S::CTAS), S::THREADS, S::SMEM, stream>>>(bp);
  return cudaGetLastError();
}
template <int DIN>
cudaError_t launch_bwd_kernel(const BwdParams& bp, int B, int H, cudaStream_t stream) {
  return bp.u_fwd ? launch_bwd_kernel<DIN, true>(bp, B, H, stream)
                  : launch_bwd_kernel<DIN, false>(bp, B, H, stream);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

// Workspace of the backward: the forward's own workspace, the state at every
// chunk boundary, the per-(sequence, head) scratch of one chunk's sub-block
// states, and every token's u from the forward (fp32, like an output).
size_t chunk_bwd_workspace_bytes(int B, int T, int H, int d) {
  const size_t dd = (size_t)d * d * sizeof(float);
  const size_t n_ckpt = (size_t)(T / BW_CH);
  return align256(chunk_workspace_bytes(false, B, T, H)) + align256((size_t)B * n_ckpt * H * dd) +
         align256((size_t)B * H * (BW_CH / SUB) * dd) + align256((size_t)B * T * H * d * sizeof(float));
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
  float* ufwd = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(scratch) +
                                         align256((size_t)B * H * (BW_CH / SUB) * dd));
  // the forward, for the state at every chunk boundary (its outputs are not needed)
  ChunkProblem f = fwd;
  f.out = nullptr;
  f.final_state = nullptr;
  f.ckpt = n_ckpt > 0 ? ckpt : nullptr;
  f.ckpt_every_chunks = 1;
  f.n_ckpt = n_ckpt;
  f.scan_segs = 0;
  // and every token's u where the forward can write it (then the token
  // states are rebuilt without column sums)
  f.u_out = chunk_fwd_writes_u(B, H) ? ufwd : nullptr;
  cudaError_t e = launch_chunk_fwd(f, fwd_ws, stream);
  if (e != cudaSuccess) return e;
  BwdParams bp{static_cast<const __nv_bfloat16*>(fwd.q), static_cast<const __nv_bfloat16*>(fwd.k),
               static_cast<const __nv_bfloat16*>(fwd.v), static_cast<const __nv_bfloat16*>(fwd.log_alpha),
               static_cast<const __nv_bfloat16*>(fwd.beta), fwd.initial_state, ckpt, d_out, d_final,
               dq, dk, dv, dla, dbeta, ds0, scratch, f.u_out, T, H, n_ckpt, fwd.scale};
  // dq, dk, dlog_alpha and dbeta are summed over the column blocks
  const size_t tok_bytes = (size_t)B * T * H * d * sizeof(float);
  for (float* x : {dq, dk, dla}) {
    e = cudaMemsetAsync(x, 0, tok_bytes, stream);
    if (e != cudaSuccess) return e;
  }
  e = cudaMemsetAsync(dbeta, 0, (size_t)B * T * H * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  return d == 64 ? launch_bwd_kernel<64>(bp, B, H, stream) : launch_bwd_kernel<128>(bp, B, H, stream);
}

}  // namespace kda
