// Chunked KDA prefill on tcgen05 tensor cores.
//
// One CTA (128 threads) walks one (sequence, head) through 64-token chunks
// made of four 16-token tiles.  Per chunk, with g the cumulative log-decay
// from the chunk start (per key channel, inclusive) and S the fp32 state
// entering the chunk:
//
//   A_qk[r,i] = sum_c q_rc k_ic e^{g_rc - g_ic}          (i <= r)
//   A_kk[r,i] = beta_r sum_c k_rc k_ic e^{g_rc - g_ic}   (i <  r)
//   T  = (I + A_kk)^-1,   W = T diag(beta) (k * e^g),   U~ = T diag(beta) V
//   U  = U~ - W S
//   O  = scale ((q * e^g) S + A_qk U)
//   S <- Diag(e^{g_C}) S + (k * e^{g_C - g})^T U
//
// This is the blockwise evaluation that, per the orkas.ai page ("Kimi K3
// architecture", section "Eine Untergrenze, die einen GPU-Codepfad
// beseitigte"), has to divide by the accumulated decay.  With log_alpha in
// [-5, 0], the log-decay across a 16-token tile spans at most 80, so for a
// column tile b with end reference E_b = g at its last token,
//   e^{g_r - g_i} = e^{g_r - E_b} * e^{E_b - g_i},   i in tile b, r >= i,
// has a left factor in [0, e^80] and a right factor in [e^-80, 1]: both fit
// bf16/fp32.  So the DIAGONAL tiles use the same dense bf16 tcgen05 product
// as the off-diagonal ones; there is no per-position-pair special path.
//
// Every product is a tcgen05.mma with M = 128 (fp32 accumulators in TMEM):
//   M1 (x4) [Q^(b); K^(b)] (128 x d) . Kb[tile b]^T      -> A_qk | A_kk column tile b
//   M2      (k e^g)^T (d x 64) . (T diag beta)^T        -> W^T
//   M3      V^T . (T diag beta)^T                       -> U~^T
//   M4      U^T  = U~^T - S^T W^T                       (negated A operand)
//   M5      O^T  = S^T (q e^g)^T + U^T A_qk^T
//   M6      S^T <- S^T Diag(e^{g_C}) + U^T K-bar
// The state is kept transposed (S^T, value channel = TMEM lane) in TMEM as
// an fp32 accumulator; its 16-bit copy in shared memory is the MMA operand.
//
// Precision.  The tile-referenced M1 operands span e^{+-80} and need bf16's
// range; their 8-bit mantissa alone costs too much accuracy in A, so each is
// split into a bf16 pair x = hi + lo and M1 accumulates hi.hi + lo.hi + hi.lo
// (three MMAs per tile, fp32 accumulation).  Every state-pass operand (S, W,
// q e^g, U, A_qk, k e^{g_C - g}) is bounded by O(1)..O(10) and is stored as
// fp16 (3 more mantissa bits than bf16, same tensor-core rate).  The M2/M3
// operands pair with the raw bf16 v tile and stay bf16.
// The 64x64 unit lower-triangular inverse is formed in fp32 on CUDA cores
// (16x16 diagonal blocks by forward substitution, then block products).
//
// d = 64 heads run the d = 128 code with the upper channel half zeroed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tma_host.h"
#include "umma.cuh"

namespace kda {

static __device__ int g_chunk_status = 0;

namespace {

constexpr int CH = 64;   // tokens per chunk
constexpr int DP = 128;  // padded head dimension
constexpr int NTHREADS = 128;
constexpr float LOG2E = 1.4426950408889634f;

// Shared-memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_RQ = 0;        // raw q tile  [64 tok][128 ch], TMA, 128B swizzle
constexpr uint32_t OFF_RK = 16384;    // raw k tile
constexpr uint32_t OFF_RG = 32768;    // raw log_alpha tile
constexpr uint32_t OFF_RV = 49152;    // raw v tile (also the V^T operand of M3)
constexpr uint32_t OFF_XH = 65536;    // M1 A operand of the current tile version, hi part
constexpr uint32_t OFF_XL = 98304;    // ... lo part
constexpr uint32_t OFF_KT = 65536;    // (k e^g)^T          (after M1)
constexpr uint32_t OFF_QT = 81920;    // (q e^g)            (after M1)
constexpr uint32_t OFF_KBAR = 98304;  // k e^{g_C - g}       (after M1)
constexpr uint32_t OFF_AKK = 114688;  // A_kk fp32 [64][64]  (after M1)
constexpr uint32_t OFF_KB = 131072;   // M1 B operand: k e^{E_b - g}, hi part
constexpr uint32_t OFF_KBL = 188416;  // ... lo part (shares the U^T buffer, free during M1)
constexpr uint32_t OFF_WT = 131072;   // W (fp16)            (after M1)
constexpr uint32_t OFF_TB = 147456;   // T diag(beta) (bf16)
constexpr uint32_t OFF_ST = 155648;   // S^T (fp16), 2 K-blocks
constexpr uint32_t OFF_UT = 188416;   // U^T (fp16)
constexpr uint32_t OFF_AQ = 204800;   // A_qk (fp16)
constexpr uint32_t OFF_TI = 212992;   // T fp32 [64][64]
constexpr uint32_t SMEM_BYTES = 229376 + 1024;

// TMEM columns.
constexpr uint32_t TM_A = 0, TM_W = 64, TM_U = 128, TM_O = 192, TM_S = 256, TM_COLS = 512;

struct Params {
  const __nv_bfloat16* beta;
  const float* s0;
  void* out;
  float* s1;
  const int* cu;  // device cu_seqlens (packed) or null (fixed length)
  int T;          // tokens per sequence when cu is null
  int H;
  float scale;
  int check_decay;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ OperandLayout kmajor(uint32_t base, uint32_t kb_stride) {
  OperandLayout L;
  L.base = base;
  L.sw = SW_128;
  L.mn_major = false;
  L.lbo = 0;
  L.sbo = 1024;
  L.kb_stride = kb_stride;
  return L;
}
__device__ __forceinline__ OperandLayout mnmajor(uint32_t base, uint32_t lbo) {
  OperandLayout L;
  L.base = base;
  L.sw = SW_128;
  L.mn_major = true;
  L.lbo = lbo;
  L.sbo = 1024;
  L.kb_stride = 0;
  return L;
}

// 8 consecutive bf16 / fp16 values (16 bytes) at a swizzled address.
__device__ __forceinline__ void st8(uint32_t addr, const float* x) {
  st_shared_v4(addr, pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
               pack_bf16x2(x[6], x[7]));
}
__device__ __forceinline__ void st8h(uint32_t addr, const float* x) {
  st_shared_v4(addr, pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
               pack_f16x2(x[6], x[7]));
}
// x as an unevaluated bf16 pair: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(const float* x, float* hi, float* lo) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    hi[j] = __bfloat162float(__float2bfloat16_rn(x[j]));
    lo[j] = x[j] - hi[j];
  }
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  float a[16], b[16], c[16], d[16];
  tmem_ld16(taddr, a);
  tmem_ld16(taddr + 16, b);
  tmem_ld16(taddr + 32, c);
  tmem_ld16(taddr + 48, d);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = a[i];
    v[16 + i] = b[i];
    v[32 + i] = c[i];
    v[48 + i] = d[i];
  }
}

// Version b of the M1 A operand: rows r >= 16 b of [Q^(b); K^(b)] with
// Q^(b)_rc = q_rc e^{g_rc - E_bc} = q_rc p_r F[tile(r)][b] (same for K).
// Rows above 16 b are never read back (their products are masked).
template <int B>
__device__ __forceinline__ void build_version(const OperandLayout& LXh, const OperandLayout& LXl,
                                              const OperandLayout& LQ, const OperandLayout& LK,
                                              int c, int valid, const float (&p)[CH],
                                              const float (&F)[4][4]) {
#pragma unroll
  for (int r0 = 16 * B; r0 < CH; r0 += 8) {
    float fq[8], fk[8], hi[8], lo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = r0 + j;
      const float f = p[r] * F[r / 16][B];
      const bool ok = r < valid;
      fq[j] = ok ? bf2f(ld_shared_u16(layout_addr(LQ, r, c))) * f : 0.f;
      fk[j] = ok ? bf2f(ld_shared_u16(layout_addr(LK, r, c))) * f : 0.f;
    }
    split_bf16(fq, hi, lo);
    st8(layout_addr(LXh, r0, c), hi);
    st8(layout_addr(LXl, r0, c), lo);
    split_bf16(fk, hi, lo);
    st8(layout_addr(LXh, CH + r0, c), hi);
    st8(layout_addr(LXl, CH + r0, c), lo);
  }
}

template <int DIN, typename OutT>
__global__ void __launch_bounds__(NTHREADS, 1)
    kda_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                     Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t tma_bar, mma_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ float s_beta[CH];
  __shared__ float s_gamma[DP];
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.x, n = blockIdx.y;
  const int H = p.H;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sbp = smem_raw + (sb - raw);

  int tok0, len;
  if (p.cu) {
    tok0 = p.cu[n];
    len = p.cu[n + 1] - tok0;
  } else {
    tok0 = n * p.T;
    len = p.T;
  }
  const int nchunks = len > 0 ? (len + CH - 1) / CH : 0;

  const OperandLayout L_RQ = kmajor(sb + OFF_RQ, 8192), L_RK = kmajor(sb + OFF_RK, 8192);
  const OperandLayout L_RG = kmajor(sb + OFF_RG, 8192);
  const OperandLayout L_VA = mnmajor(sb + OFF_RV, 8192);   // M = v, K = i
  const OperandLayout L_XH = mnmajor(sb + OFF_XH, 16384);  // M = [q r; k r], K = c
  const OperandLayout L_XL = mnmajor(sb + OFF_XL, 16384);
  const OperandLayout L_KB = mnmajor(sb + OFF_KB, 16384);   // N = i, K = c
  const OperandLayout L_KBL = mnmajor(sb + OFF_KBL, 16384);
  const OperandLayout L_TB = kmajor(sb + OFF_TB, 0);       // N = r, K = i
  const OperandLayout L_KT = kmajor(sb + OFF_KT, 0);       // M = c, K = i
  const OperandLayout L_QT = mnmajor(sb + OFF_QT, 16384);  // N = r, K = c
  const OperandLayout L_WT = mnmajor(sb + OFF_WT, 16384);  // N = r, K = c
  const OperandLayout L_KBAR = kmajor(sb + OFF_KBAR, 0);   // N = c, K = i
  const OperandLayout L_ST = kmajor(sb + OFF_ST, 16384);   // M = v, K = c
  const OperandLayout L_UT = kmajor(sb + OFF_UT, 0);       // M = v, K = i
  const OperandLayout L_AQ = kmajor(sb + OFF_AQ, 0);       // N = r, K = i
  float* akk = reinterpret_cast<float*>(sbp + OFF_AKK);
  float* ti = reinterpret_cast<float*>(sbp + OFF_TI);

  if (tid == 0) {
    mbar_init(&tma_bar, 1);
    mbar_init(&mma_bar, 1);
    mbar_fence_init();
    s_abort = 0;
  }
  if (DIN == 64) {  // the upper channel half of every raw tile stays zero
    for (uint32_t off = tid * 16; off < 8192; off += NTHREADS * 16) {
      st_shared_v4(sb + OFF_RQ + 8192 + off, 0, 0, 0, 0);
      st_shared_v4(sb + OFF_RK + 8192 + off, 0, 0, 0, 0);
      st_shared_v4(sb + OFF_RG + 8192 + off, 0, 0, 0, 0);
      st_shared_v4(sb + OFF_RV + 8192 + off, 0, 0, 0, 0);
    }
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's 32 TMEM lanes

  uint32_t tma_phase = 0, mma_phase = 0;
  bool tma_pending = false;
  constexpr uint32_t kTxBytes = 4u * (DIN / 64) * 8192u;
  auto issue_loads = [&](int chunk) {
    const int t = tok0 + chunk * CH;
    mbar_arrive_expect_tx(&tma_bar, kTxBytes);
#pragma unroll
    for (int b = 0; b < DIN / 64; ++b) {
      tma_load_3d(sbp + OFF_RQ + b * 8192, &tm_q, &tma_bar, b * 64, h, t);
      tma_load_3d(sbp + OFF_RK + b * 8192, &tm_k, &tma_bar, b * 64, h, t);
      tma_load_3d(sbp + OFF_RG + b * 8192, &tm_g, &tma_bar, b * 64, h, t);
      tma_load_3d(sbp + OFF_RV + b * 8192, &tm_v, &tma_bar, b * 64, h, t);
    }
  };
  if (nchunks > 0) {
    if (tid == 0) issue_loads(0);
    tma_pending = true;
  }

  // Bounded wait on a barrier by every thread; a timeout anywhere aborts the CTA.
  auto wait_all = [&](uint64_t* bar, uint32_t& phase) -> bool {
    const bool ok = mbar_wait(bar, phase);
    if (!ok) {
      s_abort = 1;
      atomicExch(&g_chunk_status, 6);
    }
    phase ^= 1u;
    __syncthreads();
    tc_fence_after_sync();
    return s_abort == 0;
  };
  // Make this thread's smem operand writes visible to the tensor core and
  // meet the other threads before thread 0 issues MMAs.
  auto operands_ready = [&]() {
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
  };

  // Initial state: thread v holds row v of S^T.
  {
    const int v = tid;
    const size_t sbase = (size_t)(n * H + h) * DIN * DIN;
#pragma unroll
    for (int c0 = 0; c0 < DP; c0 += 16) {
      float s[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j;
        s[j] = (p.s0 && c < DIN && v < DIN) ? p.s0[sbase + (size_t)c * DIN + v] : 0.f;
      }
      tmem_st16(tl + TM_S + c0, s);
      st8h(layout_addr(L_ST, v, c0), s);
      st8h(layout_addr(L_ST, v, c0 + 8), s + 8);
    }
    tmem_st_wait();
  }

  constexpr uint32_t ID_M1 = make_idesc(128, 16, true, true);                // bf16
  constexpr uint32_t ID_W = make_idesc(128, 64, false, false);               // bf16
  constexpr uint32_t ID_V = make_idesc(128, 64, true, false);                // bf16
  constexpr uint32_t ID_U = make_idesc(128, 64, false, true, true, true);    // fp16, -A
  constexpr uint32_t ID_O1 = make_idesc(128, 64, false, true, false, true);  // fp16
  constexpr uint32_t ID_O2 = make_idesc(128, 64, false, false, false, true); // fp16
  constexpr uint32_t ID_S = make_idesc(128, 128, false, false, false, true); // fp16

  const int c = tid;  // key channel owned in the elementwise stages
  for (int chunk = 0; chunk < nchunks; ++chunk) {
    const int t0 = tok0 + chunk * CH;
    const int valid = min(CH, len - chunk * CH);

    if (tid < CH) s_beta[tid] = tid < valid ? __bfloat162float(p.beta[(size_t)(t0 + tid) * H + h]) : 0.f;
    if (!wait_all(&tma_bar, tma_phase)) break;
    tma_pending = false;

    // ---- cumulative log-decay and per-tile references (thread = channel c)
    float pr[CH];  // p_r = e^{g_r - E_tile(r)} in [1, e^80]
    float E[4];
    {
      float acc = 0.f;
      bool bad = false;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        float la = bf2f(ld_shared_u16(layout_addr(L_RG, i, c)));
        la = i < valid ? la : 0.f;
        bad |= !(la >= -5.f && la <= 0.f);
        acc += la;
        pr[i] = acc;
      }
      if (p.check_decay && bad) atomicExch(&g_chunk_status, 5);
#pragma unroll
      for (int b = 0; b < 4; ++b) E[b] = pr[16 * b + 15];
#pragma unroll
      for (int i = 0; i < CH; ++i) pr[i] = ex2((pr[i] - E[i / 16]) * LOG2E);
    }
    float F[4][4];  // F[a][b] = e^{E_a - E_b} (a >= b)
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) F[a][b] = a > b ? ex2((E[a] - E[b]) * LOG2E) : 1.f;
    float GE[4];  // e^{E_a}
#pragma unroll
    for (int a = 0; a < 4; ++a) GE[a] = ex2(E[a] * LOG2E);

    // ---- M1: column tile b of [A_qk; A_kk] = [Q^(b); K^(b)] . Kb[tile b]^T, with
    // each factor as a bf16 pair (hi.hi + lo.hi + hi.lo), one tile version at a time
#pragma unroll
    for (int i0 = 0; i0 < CH; i0 += 8) {
      float fk[8], hi[8], lo[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + j;
        fk[j] = i < valid ? bf2f(ld_shared_u16(layout_addr(L_RK, i, c))) * rcp(pr[i]) : 0.f;
      }
      split_bf16(fk, hi, lo);
      st8(layout_addr(L_KB, i0, c), hi);
      st8(layout_addr(L_KBL, i0, c), lo);
    }
    bool m1_ok = true;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (b == 0) build_version<0>(L_XH, L_XL, L_RQ, L_RK, c, valid, pr, F);
      if (b == 1) build_version<1>(L_XH, L_XL, L_RQ, L_RK, c, valid, pr, F);
      if (b == 2) build_version<2>(L_XH, L_XL, L_RQ, L_RK, c, valid, pr, F);
      if (b == 3) build_version<3>(L_XH, L_XL, L_RQ, L_RK, c, valid, pr, F);
      operands_ready();
      if (tid == 0) {
        const uint32_t d = tmem + TM_A + 16 * b;
#pragma unroll
        for (int k0 = 0; k0 < DP; k0 += 16) {
          umma_bf16(d, layout_desc(L_XH, 0, k0), layout_desc(L_KB, 16 * b, k0), ID_M1, k0 > 0);
          umma_bf16(d, layout_desc(L_XL, 0, k0), layout_desc(L_KB, 16 * b, k0), ID_M1, 1);
          umma_bf16(d, layout_desc(L_XH, 0, k0), layout_desc(L_KBL, 16 * b, k0), ID_M1, 1);
        }
        umma_commit(&mma_bar);
      }
      if (!wait_all(&mma_bar, mma_phase)) {
        m1_ok = false;
        break;
      }
    }
    if (!m1_ok) break;

    // ---- A_qk (fp16 operand) and beta-scaled strictly-lower A_kk (fp32)
    {
      float a[64];
      tmem_ld64(tl + TM_A, a);
      if (warp < 2) {
        const int r = tid;
#pragma unroll
        for (int i0 = 0; i0 < CH; i0 += 8) {
          float x[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) x[j] = (i0 + j <= r) ? a[i0 + j] : 0.f;
          st8h(layout_addr(L_AQ, r, i0), x);
        }
      } else {
        const int r = tid - CH;
        const float br = s_beta[r];
        float4* row = reinterpret_cast<float4*>(akk + r * CH);
#pragma unroll
        for (int i0 = 0; i0 < CH; i0 += 4) {
          float4 x;
          x.x = (i0 + 0 < r) ? br * a[i0 + 0] : 0.f;
          x.y = (i0 + 1 < r) ? br * a[i0 + 1] : 0.f;
          x.z = (i0 + 2 < r) ? br * a[i0 + 2] : 0.f;
          x.w = (i0 + 3 < r) ? br * a[i0 + 3] : 0.f;
          row[i0 / 4] = x;
        }
      }
    }
    // ---- state-pass operands (thread = channel c): (k e^g)^T, q e^g, k e^{g_C - g}
#pragma unroll
    for (int i0 = 0; i0 < CH; i0 += 8) {
      float kt[8], qt[8], kb[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + j, a = i / 16;
        const bool ok = i < valid;
        const float kv = ok ? bf2f(ld_shared_u16(layout_addr(L_RK, i, c))) : 0.f;
        const float qv = ok ? bf2f(ld_shared_u16(layout_addr(L_RQ, i, c))) : 0.f;
        const float gam = pr[i] * GE[a];
        kt[j] = kv * gam;
        qt[j] = qv * gam;
        kb[j] = kv * rcp(pr[i]) * F[3][a];
      }
      st8(layout_addr(L_KT, c, i0), kt);     // bf16: pairs with T diag(beta)
      st8h(layout_addr(L_QT, i0, c), qt);
      st8h(layout_addr(L_KBAR, c, i0), kb);
    }
    s_gamma[c] = GE[3];
    __syncthreads();

    // ---- T = (I + A_kk)^-1: diagonal 16x16 blocks by forward substitution
    if (tid < 64) {
      const int a = tid >> 4, j = tid & 15;
      float x[16];
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) x[rr] = rr == j ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float xm = x[m];
#pragma unroll
        for (int rr = m + 1; rr < 16; ++rr) x[rr] -= akk[(16 * a + rr) * CH + 16 * a + m] * xm;
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) ti[(16 * a + rr) * CH + 16 * a + j] = x[rr];
    }
    __syncthreads();
    // ---- off-diagonal blocks: T_ab = -T_aa sum_{m=b}^{a-1} L_am T_mb, by distance a - b
#pragma unroll 1
    for (int s = 1; s < 4; ++s) {
      const int nel = (4 - s) * 256;
      for (int e = tid; e < nel; e += NTHREADS) {
        const int b = e >> 8, a = b + s, rr = (e >> 4) & 15, cc = e & 15;
        float acc = 0.f;
        for (int m = b; m < a; ++m)
#pragma unroll
          for (int x = 0; x < 16; ++x)
            acc += akk[(16 * a + rr) * CH + 16 * m + x] * ti[(16 * m + x) * CH + 16 * b + cc];
        ti[(16 * b + rr) * CH + 16 * a + cc] = acc;  // scratch in the (zero) upper triangle
      }
      __syncthreads();
      for (int e = tid; e < nel; e += NTHREADS) {
        const int b = e >> 8, a = b + s, rr = (e >> 4) & 15, cc = e & 15;
        float acc = 0.f;
        for (int x = 0; x <= rr; ++x)
          acc += ti[(16 * a + rr) * CH + 16 * a + x] * ti[(16 * b + x) * CH + 16 * a + cc];
        ti[(16 * a + rr) * CH + 16 * b + cc] = -acc;
      }
      __syncthreads();
    }
    // ---- T diag(beta) in bf16 (rows r, K = i), lower triangle only
    {
      const int r = tid >> 1, i_lo = (tid & 1) * 32;
#pragma unroll
      for (int i0 = i_lo; i0 < i_lo + 32; i0 += 8) {
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j;
          x[j] = i <= r ? ti[r * CH + i] * s_beta[i] : 0.f;
        }
        st8(layout_addr(L_TB, r, i0), x);
      }
    }
    operands_ready();
    if (tid == 0) {
#pragma unroll
      for (int k0 = 0; k0 < CH; k0 += 16) {
        umma_bf16(tmem + TM_W, layout_desc(L_KT, 0, k0), layout_desc(L_TB, 0, k0), ID_W, k0 > 0);
        umma_bf16(tmem + TM_U, layout_desc(L_VA, 0, k0), layout_desc(L_TB, 0, k0), ID_V, k0 > 0);
      }
      umma_commit(&mma_bar);
    }
    if (!wait_all(&mma_bar, mma_phase)) break;
    // raw tiles are consumed: fetch the next chunk while the state pass runs
    if (chunk + 1 < nchunks) {
      if (tid == 0) {
        fence_proxy_async_smem();
        issue_loads(chunk + 1);
      }
      tma_pending = true;
    }

    // ---- W (fp16, N = r, K = c) from W^T in TMEM (lane = c)
    {
      float w[64];
      tmem_ld64(tl + TM_W, w);
#pragma unroll
      for (int r0 = 0; r0 < CH; r0 += 8) st8h(layout_addr(L_WT, r0, c), w + r0);
    }
    operands_ready();
    if (tid == 0) {
#pragma unroll
      for (int k0 = 0; k0 < DP; k0 += 16) {
        umma_bf16(tmem + TM_U, layout_desc(L_ST, 0, k0), layout_desc(L_WT, 0, k0), ID_U, 1);
        umma_bf16(tmem + TM_O, layout_desc(L_ST, 0, k0), layout_desc(L_QT, 0, k0), ID_O1, k0 > 0);
      }
      umma_commit(&mma_bar);
    }
    if (!wait_all(&mma_bar, mma_phase)) break;

    // ---- U^T (fp16 operand) and the chunk decay of the fp32 state
    {
      const int v = tid;
      float u[64];
      tmem_ld64(tl + TM_U, u);
#pragma unroll
      for (int r0 = 0; r0 < CH; r0 += 8) st8h(layout_addr(L_UT, v, r0), u + r0);
#pragma unroll
      for (int c0 = 0; c0 < DP; c0 += 16) {
        float s[16];
        tmem_ld16(tl + TM_S + c0, s);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) s[j] *= s_gamma[c0 + j];
        tmem_st16(tl + TM_S + c0, s);
      }
      tmem_st_wait();
    }
    operands_ready();
    if (tid == 0) {
#pragma unroll
      for (int k0 = 0; k0 < CH; k0 += 16) {
        umma_bf16(tmem + TM_O, layout_desc(L_UT, 0, k0), layout_desc(L_AQ, 0, k0), ID_O2, 1);
        umma_bf16(tmem + TM_S, layout_desc(L_UT, 0, k0), layout_desc(L_KBAR, 0, k0), ID_S, 1);
      }
      umma_commit(&mma_bar);
    }
    if (!wait_all(&mma_bar, mma_phase)) break;

    // ---- outputs and the fp16 state operand for the next chunk (thread = value channel)
    {
      const int v = tid;
      float o[64];
      tmem_ld64(tl + TM_O, o);
      if (v < DIN) {
        OutT* out = static_cast<OutT*>(p.out) + (size_t)t0 * H * DIN + (size_t)h * DIN + v;
#pragma unroll
        for (int r = 0; r < CH; ++r)
          if (r < valid) store_out(out + (size_t)r * H * DIN, p.scale * o[r]);
      }
#pragma unroll
      for (int c0 = 0; c0 < DP; c0 += 16) {
        float s[16];
        tmem_ld16(tl + TM_S + c0, s);
        tmem_ld_wait();
        st8h(layout_addr(L_ST, v, c0), s);
        st8h(layout_addr(L_ST, v, c0 + 8), s + 8);
      }
    }
  }

  if (s_abort == 0 && p.s1) {  // final state from the fp32 accumulator: S[c][v] = S^T[v][c]
    const int v = tid;
    const size_t sbase = (size_t)(n * H + h) * DIN * DIN;
#pragma unroll
    for (int c0 = 0; c0 < DP; c0 += 16) {
      float s[16];
      tmem_ld16(tl + TM_S + c0, s);
      tmem_ld_wait();
      if (v < DIN)
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < DIN) p.s1[sbase + (size_t)(c0 + j) * DIN + v] = s[j];
    }
  }
  if (s_abort && tma_pending) mbar_wait(&tma_bar, tma_phase);  // let an issued copy land
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

template <int DIN, typename OutT>
cudaError_t launch_variant(const ChunkProblem& pr, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& tg, const Params& prm,
                           cudaStream_t stream) {
  auto kern = kda_chunk_kernel<DIN, OutT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((unsigned)pr.H, (unsigned)pr.n_seq);
  kern<<<grid, NTHREADS, SMEM_BYTES, stream>>>(tq, tk, tv, tg, prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_fwd(const ChunkProblem& pr, cudaStream_t stream) {
  const uint64_t d = (uint64_t)pr.d, H = (uint64_t)pr.H;
  if (pr.T_total == 0) {
    // no tokens at all: the final state is the initial state
    if (!pr.final_state) return cudaSuccess;
    const size_t bytes = (size_t)pr.n_seq * pr.H * pr.d * pr.d * sizeof(float);
    if (pr.initial_state)
      return pr.initial_state == pr.final_state
                 ? cudaSuccess
                 : cudaMemcpyAsync(pr.final_state, pr.initial_state, bytes,
                                   cudaMemcpyDeviceToDevice, stream);
    return cudaMemsetAsync(pr.final_state, 0, bytes, stream);
  }
  const uint64_t rows = (uint64_t)pr.T_total;
  CUtensorMap tq, tk, tv, tg;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_map_3d_bf16(&tq, pr.q, d, H, rows, d, H * d, 64, 1, 64, sw) ||
      !make_map_3d_bf16(&tk, pr.k, d, H, rows, d, H * d, 64, 1, 64, sw) ||
      !make_map_3d_bf16(&tv, pr.v, d, H, rows, d, H * d, 64, 1, 64, sw) ||
      !make_map_3d_bf16(&tg, pr.log_alpha, d, H, rows, d, H * d, 64, 1, 64, sw))
    return cudaErrorInvalidValue;
  Params prm{static_cast<const __nv_bfloat16*>(pr.beta), pr.initial_state, pr.out,
             pr.final_state, pr.cu_seqlens, pr.T, pr.H, pr.scale, pr.check_decay ? 1 : 0};
  if (pr.d == 128)
    return pr.out_f32 ? launch_variant<128, float>(pr, tq, tk, tv, tg, prm, stream)
                      : launch_variant<128, __nv_bfloat16>(pr, tq, tk, tv, tg, prm, stream);
  return pr.out_f32 ? launch_variant<64, float>(pr, tq, tk, tv, tg, prm, stream)
                    : launch_variant<64, __nv_bfloat16>(pr, tq, tk, tv, tg, prm, stream);
}

int read_and_clear_chunk_status(cudaStream_t stream, cudaError_t* err) {
  int h = 0, zero = 0;
  *err = cudaStreamSynchronize(stream);
  if (*err != cudaSuccess) return 0;
  *err = cudaMemcpyFromSymbol(&h, g_chunk_status, sizeof(int));
  if (*err != cudaSuccess) return 0;
  *err = cudaMemcpyToSymbol(g_chunk_status, &zero, sizeof(int));
  return h;
}

}  // namespace kda
