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
// token's u; one CTA per (sequence, head, block of 8 value columns) then
// walks the chunks from last to first.  For each chunk it rebuilds the token
// states in fp32 from the saved chunk-start state: with u given that is a
// local step per token (S'_t = Diag(alpha_t) S_{t-1}, S_t = S'_t + k_t u_t^T,
// w_t = u_t / beta_t), and only without it, or for a token with beta = 0,
// does w take a column sum.  It keeps the state before every 4th token (in a
// per-CTA scratch in global memory) and, in the reverse recurrence, rebuilds
// each group of 4 token states in registers from it.  Thread c holds row c of
// G for the block's columns in registers: dot products along a row stay in
// the thread, sums down a column (du, and w without u) take a warp
// reduce-scatter and one pass over shared memory.  This is CUDA-core work,
// serial in tokens per (sequence, head): an exact token-level formulation,
// not a tensor-core one.
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
  float* scratch;      // [B * H][64 / SUB][d][d]
  const float* u_fwd;  // [B][T][H][d]: every token's u from the forward (HAVE_U), or null
  int T, H, n_ckpt;
  float scale;
};

// One CTA per (sequence, head, block of CB value columns): the columns of G
// evolve independently (each step scales rows and adds rank-one terms), so
// only the gradients summed along a row (dq, dk, dlog_alpha, dbeta) combine
// the blocks, by atomic adds into zeroed buffers.  Thread c owns key row c
// and the block's CB columns.
constexpr int CB = 8;
// Tokens per sub-block of the reverse pass: the state before each sub-block
// is saved (in the per-CTA scratch), and the sub-block's token states are
// rebuilt in registers when the reverse pass reaches it.
constexpr int SUB = 4;

template <int DIN>
struct BwdShape {
  static constexpr int THREADS = DIN;  // one thread per key row
  static constexpr int WARPS = THREADS / 32;
  static constexpr int BLOCKS = DIN / CB;
  // shared memory: q, k, log alpha (bf16, every channel), the block's v
  // (bf16), do, u, w (fp32), the column-sum partials, one vector, beta
  static constexpr size_t OFF_Q = 0;
  static constexpr size_t OFF_K = OFF_Q + BW_CH * DIN * 2;
  static constexpr size_t OFF_LA = OFF_K + BW_CH * DIN * 2;
  static constexpr size_t OFF_V = OFF_LA + BW_CH * DIN * 2;
  static constexpr size_t OFF_DO = OFF_V + BW_CH * CB * 2;
  static constexpr size_t OFF_U = OFF_DO + BW_CH * CB * 4;
  static constexpr size_t OFF_W = OFF_U + BW_CH * CB * 4;
  static constexpr size_t OFF_RED = OFF_W + BW_CH * CB * 4;
  static constexpr size_t OFF_VEC = OFF_RED + WARPS * CB * 4;
  static constexpr size_t OFF_BETA = OFF_VEC + CB * 4;
  static constexpr size_t SMEM = OFF_BETA + BW_CH * 4;
};

__device__ __forceinline__ float bfv(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

// Sum of x over the warp's 32 rows for each of the CB columns: a
// reduce-scatter over lane bits 4, 3, .. (one halving per bit, log2 CB
// steps) leaves the lanes that differ only in the remaining low bits with
// partial sums of one column, which a few exchanges add; the first of them
// writes red[warp][column].  The caller synchronises and adds the warps.
static_assert(CB == 8 || CB == 16 || CB == 32, "column blocks of 8, 16 or 32");
constexpr int LOG_CB = CB == 8 ? 3 : CB == 16 ? 4 : 5;
__device__ __forceinline__ void column_partials(float (&x)[CB], float* red, int warp, int lane) {
#pragma unroll
  for (int step = 0; step < LOG_CB; ++step) {
    const int bit = 16 >> step;         // lane bit 4, 3, ...
    const int half = CB >> (step + 1);  // values kept after this step
    const bool up = (lane & bit) != 0;  // keep the upper half of the current range
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? x[i] : x[i + half];
      float keep = up ? x[i + half] : x[i];
      keep += __shfl_xor_sync(0xffffffffu, send, bit);
      x[i] = keep;
    }
  }
  constexpr int LOW = 5 - LOG_CB;  // lane bits left: the same column on 2^LOW lanes
#pragma unroll
  for (int o = 1; o < (1 << LOW); o <<= 1) x[0] += __shfl_xor_sync(0xffffffffu, x[0], o);
  if ((lane & ((1 << LOW) - 1)) == 0) red[warp * CB + (lane >> LOW)] = x[0];
}

// HAVE_U: the forward left every token's u, so the chunk's token states
// follow from the saved chunk-start state with no column sums (w = u / beta;
// only a token with beta = 0 takes the sum for its w).
template <int DIN, bool HAVE_U>
__global__ void __launch_bounds__(BwdShape<DIN>::THREADS) kda_bwd_kernel(BwdParams p) {
  using S = BwdShape<DIN>;
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
  const int c = tid;  // key row
  const int h = blockIdx.x, n = blockIdx.y, blk = blockIdx.z, vb = CB * blk;  // first column
  const int H = p.H, T = p.T;
  const size_t dd = (size_t)DIN * DIN;
  const size_t plane = ((size_t)n * H + h) * dd;     // this (sequence, head) in [B][H][d][d]
  const size_t row = plane + (size_t)c * DIN + vb;  // element (c, vb)
  // per-thread scratch of one chunk: the state before each sub-block, this
  // thread's CB values
  float* scratch = p.scratch + (((size_t)n * H + h) * S::BLOCKS + blk) * (BW_CH / SUB) * DIN * CB +
                   (size_t)tid * CB;

  auto load_row = [&](const float* src, float (&x)[CB]) {  // x = src[c][vb .. vb + CB)
#pragma unroll
    for (int j = 0; j < CB; j += 4) {
      const float4 f = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      x[j] = f.x;
      x[j + 1] = f.y;
      x[j + 2] = f.z;
      x[j + 3] = f.w;
    }
  };
  float g[CB];  // G[c][vb ..]: the gradient of the state after the current token
  load_row(p.dfin ? p.dfin + row : nullptr, g);

  const int nch = (T + BW_CH - 1) / BW_CH;
  for (int ch = nch - 1; ch >= 0; --ch) {
    const int t0 = ch * BW_CH, L = min(BW_CH, T - t0);
    // ---- stage the chunk's token rows
    __syncthreads();  // the previous chunk is done with shared memory
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
    for (int e = tid; e < BW_CH * CB / 8; e += S::THREADS) {  // the block's v columns
      const int i = e / (CB / 8), c8 = (e % (CB / 8)) * 8;
      uint4 z = make_uint4(0, 0, 0, 0);
      if (i < L) z = *reinterpret_cast<const uint4*>(p.v + (((size_t)n * T + t0 + i) * H + h) * DIN + vb + c8);
      *reinterpret_cast<uint4*>(sv + i * CB + c8) = z;
    }
    for (int e = tid; e < BW_CH * CB / 4; e += S::THREADS) {  // the block's do (and u) columns
      const int i = e / (CB / 4), c4 = (e % (CB / 4)) * 4;
      const size_t off = (((size_t)n * T + t0 + i) * H + h) * DIN + vb + c4;
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f), zu = z;
      if (i < L) {
        z = *reinterpret_cast<const float4*>(p.dout + off);
        if (HAVE_U) zu = *reinterpret_cast<const float4*>(p.u_fwd + off);
      }
      *reinterpret_cast<float4*>(sdo + i * CB + c4) = z;
      if (HAVE_U) *reinterpret_cast<float4*>(su + i * CB + c4) = zu;
    }
    if (tid < BW_CH) sbeta[tid] = tid < L ? bfv(p.beta, ((size_t)n * T + t0 + tid) * H + h) : 0.f;
    __syncthreads();

    // ---- forward over the chunk from its saved starting state
    float s[CB];
    {
      const float* src = ch == 0 ? (p.s0 ? p.s0 + plane : nullptr)
                                 : p.ckpt + (((size_t)n * p.n_ckpt + (ch - 1)) * H + h) * dd;
      load_row(src ? src + (size_t)c * DIN + vb : nullptr, s);
    }
    for (int i = 0; i < L; ++i) {
      const float a = __expf(__bfloat162float(sla[i * DIN + c]));
      const float kc = __bfloat162float(sk[i * DIN + c]);
      if ((i & (SUB - 1)) == 0) {  // S_{t-1}: the state before this sub-block
        float* dst = scratch + (size_t)(i / SUB) * DIN * CB;
#pragma unroll
        for (int j = 0; j < CB; j += 4)
          *reinterpret_cast<float4*>(dst + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
      }
      float x[CB];
#pragma unroll
      for (int j = 0; j < CB; ++j) {
        s[j] *= a;  // S'_t
        x[j] = s[j] * kc;
      }
      const float b = sbeta[i];
      if (!HAVE_U || b == 0.f) {  // (with u given: the same for every thread)
        column_partials(x, red, warp, lane);
        __syncthreads();
        if (tid < CB) {  // w = v - S'^T k, u = beta w
          float acc = 0.f;
#pragma unroll
          for (int wp = 0; wp < S::WARPS; ++wp) acc += red[wp * CB + tid];
          const float w = __bfloat162float(sv[i * CB + tid]) - acc;
          sw[i * CB + tid] = w;
          su[i * CB + tid] = b * w;
        }
        __syncthreads();
      }
#pragma unroll
      for (int j = 0; j < CB; ++j) s[j] += kc * su[i * CB + j];  // S_t
    }
    if (HAVE_U) {  // w = u / beta where beta != 0
      for (int e = tid; e < L * CB; e += S::THREADS) {
        const float b = sbeta[e / CB];
        if (b != 0.f) sw[e] = su[e] / b;
      }
      __syncthreads();
    }

    // ---- the reverse recurrence over the chunk's tokens, SUB at a time: the
    // sub-block's S'_t are rebuilt in registers from the state saved before
    // it (a local step per token: u is known), whose load is issued one
    // sub-block ahead.
    const int nsub = (L + SUB - 1) / SUB;
    float nxt[CB];
    if (nsub > 0) load_row(scratch + (size_t)(nsub - 1) * DIN * CB, nxt);
    for (int sbk = nsub - 1; sbk >= 0; --sbk) {
      float spq[SUB][CB];
      {
        float st[CB];
#pragma unroll
        for (int j = 0; j < CB; ++j) st[j] = nxt[j];
        if (sbk > 0) load_row(scratch + (size_t)(sbk - 1) * DIN * CB, nxt);
#pragma unroll
        for (int q = 0; q < SUB; ++q) {
          const int i = SUB * sbk + q;
          const float a = i < L ? __expf(__bfloat162float(sla[i * DIN + c])) : 1.f;
          const float kc = i < L ? __bfloat162float(sk[i * DIN + c]) : 0.f;
#pragma unroll
          for (int j = 0; j < CB; ++j) {
            st[j] *= a;
            spq[q][j] = st[j];
            st[j] += kc * su[(i < L ? i : 0) * CB + j];
          }
        }
      }
#pragma unroll
    for (int q = SUB - 1; q >= 0; --q) {
      const int i = SUB * sbk + q;
      if (i >= L) continue;  // (the same for every thread)
      const size_t tok = ((size_t)n * T + t0 + i) * H + h;
      const float* sp = spq[q];
      const float qc = __bfloat162float(sq[i * DIN + c]);
      const float kc = __bfloat162float(sk[i * DIN + c]);
      const float a = __expf(__bfloat162float(sla[i * DIN + c]));
      const float b = sbeta[i];
      const float* dov = sdo + i * CB;
      const float* uv = su + i * CB;
      // G += scale q do^T, then du = G^T k
      float x[CB];
#pragma unroll
      for (int j = 0; j < CB; ++j) {
        g[j] += p.scale * qc * dov[j];
        x[j] = g[j] * kc;
      }
      column_partials(x, red, warp, lane);
      __syncthreads();
      if (warp == 0) {  // du, dv = beta du, and this block's share of dbeta = du . w
        float du = 0.f, xb = 0.f;
        if (lane < CB) {
#pragma unroll
          for (int wp = 0; wp < S::WARPS; ++wp) du += red[wp * CB + lane];
          svec[lane] = du;
          p.dv[tok * DIN + vb + lane] = b * du;
          xb = du * sw[i * CB + lane];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) xb += __shfl_xor_sync(0xffffffffu, xb, o);
        if (lane == 0) atomicAdd(p.dbeta + tok, xb);
      }
      __syncthreads();
      // dq = scale S_t do with S_t = S' + k u^T;  dk = G u - beta S' du;
      // dS' = G - beta k du^T;  dlog_alpha = rowsum(dS' o S')  (this block's columns)
      float xq = 0.f, xk = 0.f, xa = 0.f;
#pragma unroll
      for (int j = 0; j < CB; ++j) {
        const float du = svec[j], u = uv[j];
        xq += (sp[j] + kc * u) * dov[j];
        xk += g[j] * u - b * sp[j] * du;
        g[j] -= b * kc * du;
        xa += g[j] * sp[j];
        g[j] *= a;  // the gradient of S_{t-1}
      }
      atomicAdd(p.dq + tok * DIN + c, p.scale * xq);
      atomicAdd(p.dk + tok * DIN + c, xk);
      atomicAdd(p.dla + tok * DIN + c, xa);
    }
    }
  }
  if (p.ds0) {
#pragma unroll
    for (int j = 0; j < CB; j += 4)
      *reinterpret_cast<float4*>(p.ds0 + row + j) = make_float4(g[j], g[j + 1], g[j + 2], g[j + 3]);
  }
}

template <int DIN, bool HAVE_U>
cudaError_t launch_bwd_kernel(const BwdParams& bp, int B, int H, cudaStream_t stream) {
  using S = BwdShape<DIN>;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_kernel<DIN, HAVE_U>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
  if (e != cudaSuccess) return e;
  kda_bwd_kernel<DIN, HAVE_U>
      <<<dim3((unsigned)H, (unsigned)B, S::BLOCKS), S::THREADS, S::SMEM, stream>>>(bp);
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
