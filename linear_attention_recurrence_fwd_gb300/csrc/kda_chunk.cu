// Chunked KDA prefill on tcgen05 tensor cores, in two stages.
//
// For a 64-token chunk (four 16-token tiles) of one (sequence, head), with
// g the cumulative log-decay from the chunk start (per key channel,
// inclusive) and S the fp32 state entering the chunk:
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
// row tile a with reference R_a = g just before its first token,
//   e^{g_r - g_i} = e^{g_r - R_a} * e^{R_a - g_i},   r in tile a, i <= r,
// has a left factor in [e^-80, 1] and a right factor in [1, e^80] on the
// diagonal tile (at most 1 before it): both fit the fp32 exponent.  So the
// DIAGONAL tiles use the same dense tcgen05 product as the off-diagonal
// ones; there is no per-position-pair special path.
//
// Stage 1 (kda_intra_kernel) needs no state, so its (chunk, head) items run
// on every SM, two CTAs per SM, each loading its next item's inputs while it
// finishes the current one.  It writes a per-chunk
// record -- W, q e^g, k e^{g_C - g}, A_qk, T diag(beta) and e^{g_C} -- as
// byte images of the shared-memory operand tiles stage 2 feeds its MMAs.
// Stage 2 (kda_state_kernel) walks each (sequence, head) serially,
// double-buffering records with bulk copies and v tiles with TMA:
//   M3  U~^T = V^T (T diag beta)^T             bf16
//   M4  U^T  = U~^T - S^T W^T                  fp16 (negated A)
//   M5  O^T  = S^T (q e^g)^T + U^T A_qk^T      fp16
//   M6  S^T <- S^T Diag(e^{g_C}) + U^T K-bar   fp16
// with S^T (value channel = TMEM lane) as an fp32 TMEM accumulator and its
// fp16 copy in shared memory as the MMA operand.
//
// Stage 1 products, all tcgen05 with M = 128:
//   the cumulative sum g^T = LA^T L^T (L lower-triangular ones) and the
//   transposes q^T = Q^T I, k^T = K^T I move per-channel columns into TMEM
//   (one thread per key channel reads them back);
//   M1 (x2) K~ . [Q~; K~]^T -> A_qk^T, A_kk^T, keys on TMEM lanes: one
//   product stacks the key operands of row tiles 3 and 2 (64 + 48 keys)
//   on M, the other those of row tiles 1 and 0 (32 + 16 keys);
//   M2 (k e^g)^T (T diag beta)^T -> W^T.
// The 64x64 unit lower-triangular inverse is formed in fp32 on CUDA cores.
//
// Precision.  The tile-referenced M1 operands span e^{+-80} and need an
// 8-bit exponent; bf16's 8-bit mantissa alone costs too much accuracy in A,
// so M1 runs as kind::tf32 on fp32 operands rounded to nearest tf32 (10
// mantissa bits), K-major so that each thread (one key channel) writes one
// element per row.  Every state-pass operand (S, W, q e^g, U, A_qk,
// k e^{g_C - g}) is bounded by O(1)..O(10) and is stored as fp16 (3 more
// mantissa bits than bf16, same tensor-core rate).  T diag(beta) and
// (k e^g)^T pair with the raw bf16 v tile / each other and stay bf16.
//
// d = 64 heads run the d = 128 code with the upper channel half zeroed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <cstdlib>
#include <mutex>

#include "kda_internal.h"
#include "tma_host.h"
#include "umma.cuh"

namespace kda {

static __device__ int g_chunk_status = 0;

namespace {

constexpr int CH = 64;   // tokens per chunk
constexpr int DP = 128;  // padded head dimension
constexpr float LOG2E = 1.4426950408889634f;

// ---- per-(chunk, head) record: stage 2's shared-memory operand images
constexpr uint32_t REC_WT = 0;         // W (fp16), B operand: N = r, K = c, MN-major
constexpr uint32_t REC_QT = 16384;     // q e^g (fp16), B operand: N = r, K = c, MN-major
constexpr uint32_t REC_KBAR = 32768;   // k e^{g_C - g} (fp16), B operand: N = c, K = i
constexpr uint32_t REC_AQ = 49152;     // A_qk (fp16), B operand: N = r, K = i, MN-major
constexpr uint32_t REC_TB = 57344;     // T diag(beta) (bf16), B operand: N = r, K = i
constexpr uint32_t REC_G = 65536;      // e^{g_C} per key channel, fp32 x 128
constexpr uint32_t REC_LOAD = 66048;   // bytes copied per record
constexpr uint32_t REC_BYTES = 66560;  // record stride

// ---- stage 1 shared memory (bytes from a 1024-aligned base); phases reuse space
// raw TMA tiles (transposes), loaded during the previous item: q and k and
// the first 64 channels of log alpha where the first record stores read,
// the other 64 channels of log alpha in a region of their own (A_RG1)
constexpr uint32_t A_RQ = 16384, A_RK = 32768, A_RG = 49152;
constexpr uint32_t A_LM = 65536, A_IM = 73728;            // L, I (bf16)      (transposes)
constexpr uint32_t A_XH = 0;                              // M1 A operand, 64 KB (M1)
constexpr uint32_t A_KBH = 65536;                         // M1 B operand, 32 KB (M1)
constexpr uint32_t A_STG = 0;                             // record image [0, 64K) (after M1)
constexpr uint32_t A_AKK = 65536;                         // A_kk fp32 [64][AKS] (after M1)
constexpr uint32_t A_KT = 82944;                          // (k e^g)^T bf16      (after M1)
constexpr uint32_t A_WST = 82944;                         // W record image      (after M2)
constexpr uint32_t A_TI = 0;                              // T fp32 (in the W slot, before W)
constexpr uint32_t A_DINV = 57344;                        // T_aa transposed, 4 KB (in the T diag(beta) slot, before it)
constexpr uint32_t A_MISC = 99328;                        // barriers, beta, gamma
// A_kk row stride in floats: 68 puts the rows' float4 chunks 16 bytes apart
// in bank order, so 32 rows written at the same column and 8 columns read
// in one row are both conflict-free.
constexpr int AKS = 68;
constexpr uint32_t A_RG1 = A_MISC + 1024;                 // raw log alpha, channels 64..127
constexpr uint32_t A_RG_LBO = A_RG1 - A_RG;               // between the log alpha halves
constexpr uint32_t A_SMEM = A_RG1 + 8192 + 1024;          // + alignment slack
// Stage 1 threads: thread t owns key channel (TMEM lane) t % 128 and, in the
// per-token stages, the token tiles {0, 3} (t < 128) or {1, 2} (t >= 128);
// over the two M1 passes both halves build nine 16-row operand pieces.
constexpr int A_THREADS = 256;

// ---- stage 2 shared memory
constexpr uint32_t B_REC0 = 0, B_V0 = 66560, B_REC1 = 82944, B_V1 = 149504;
constexpr uint32_t B_ST = 165888;  // S^T fp16, 2 K-blocks
constexpr uint32_t B_UT = 198656;  // U^T fp16
constexpr uint32_t B_MISC = 215040;
constexpr uint32_t B_SMEM = B_MISC + 1024 + 1024;

// ---- TMEM columns
// Stage 1: g, q^T, k^T from the transposes; M1 pass 0 in TA_A, pass 1 in
// TA_G (g is consumed by then); W^T from M2 in TA_W.
constexpr uint32_t TA_G = 0, TA_Q = 64, TA_K = 128, TA_A = 192, TA_W = 0, TA_COLS = 256;
// Stage 2: U~ (M3 result, two buffers), D = [-S^T W^T | -O^T] (two buffers of
// 128 columns: the U correction and the output share one N = 128 product)
// and the fp32 state S^T.
constexpr uint32_t TB_UT = 0, TB_D = 128, TB_S = 384, TB_COLS = 512;

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
// x rounded to nearest tf32 (10 explicit mantissa bits), as the bit pattern
// of an fp32 whose low 13 bits are zero.
// Adding half of the dropped unit to the bit pattern rounds the magnitude to
// nearest with ties away from zero (a carry into the exponent is the correct
// rounding up); the mask clears the 13 bits the product ignores.
__device__ __forceinline__ float tf32r(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
__device__ __forceinline__ void st_f32(uint32_t addr, float x) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(x) : "memory");
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

__device__ __forceinline__ void set_status(int code) { atomicExch(&g_chunk_status, code); }

// Address of element (row, channel c) of a K-major, 128-byte-swizzled fp32
// operand: cbase = base + (c / 32) * kb_stride, cl = (c % 32) * 4.  Row
// groups of 8 are 1024 bytes apart; the swizzle XORs the 16-byte chunk
// index with row % 8.  For rows 16 a + j with j a compile-time constant the
// row-dependent terms fold to constants.
__device__ __forceinline__ uint32_t kmaj32_addr(uint32_t cbase, uint32_t cl, int row) {
  return cbase + ((uint32_t)(row >> 3) << 10) + ((uint32_t)(row & 7) << 7) +
         (cl ^ ((uint32_t)(row & 7) << 4));
}

// M1 operands of one round, kind::tf32 (fp32 rounded to nearest tf32).
// Row tile a is referenced to R_a, the log-decay just before it (E_{a-1},
// and 0 for a = 0):
//   e^{g_r - g_i} = e^{g_r - R_a} e^{R_a - g_i},   r in tile a, i <= r.
// The left factor lies in [e^-80, 1].  The right one lies in [1, e^80] for
// keys of tile a and is at most 1 for earlier keys, where it may underflow
// to zero: the exact product is then smaller still.
//   A operand, M = 128 key rows, K~^(a)_i = k_i e^{R_a - g_i}: pass 0 holds
//     row tile 3's keys 0..63 in rows 0..63 and row tile 2's keys 0..47 in
//     rows 64..111; pass 1 row tile 1's keys 0..31 in rows 0..31 and row
//     tile 0's keys 0..15 in rows 32..47.
//   B operand, N = 64 token rows, q_r e^{g_r - R_a} and k_r e^{g_r - R_a}
//     of the pass's row tiles: rows 0..15 / 16..31 q / k of the odd tile
//     (3 or 1), rows 32..47 / 48..63 q / k of the even tile (2 or 0).
// A rows left unwritten reach only TMEM lanes that are never read.  The
// calling thread writes channel c of the rows of its tiles ta[0], ta[1]
// (p: their e^{g - E}), one element per row, a warp one 128-byte line.
// E: every tile's end; Eo, Ep: the end of tile ta[s] and of the tile before
// it (0 for tile 0).
template <int R>
__device__ __forceinline__ void build_m1_pass(uint32_t abase, uint32_t bbase, uint32_t cl,
                                            uint32_t tl, const float (&p)[2][16],
                                            const float (&E)[4], const float (&Eo)[2],
                                            const float (&Ep)[2], const int (&ta)[2]) {
  constexpr int AHI = R == 0 ? 3 : 1, ALO = AHI - 1;  // the pass's row tiles
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int t = ta[s];
    if (t > AHI) continue;           // warp-uniform
    const bool rows = t >= ALO;      // t is one of the pass's row tiles
    float kv[16], qv[16];
    tmem_ld16(tl + TA_K + 16 * t, kv);
    if (rows) tmem_ld16(tl + TA_Q + 16 * t, qv);
    tmem_ld_wait();
    const float et = Eo[s];
    const float f_hi = ex2((E[AHI - 1] - et) * LOG2E);                   // e^{R_AHI - E_t}
    const float f_lo = ex2(((ALO > 0 ? E[ALO - 1] : 0.f) - et) * LOG2E);  // e^{R_ALO - E_t}
    const float f_b = ex2((et - Ep[s]) * LOG2E);                          // e^{E_t - R_t}
    const uint32_t a_hi = abase + ((uint32_t)t << 11);
    const uint32_t a_lo = abase + ((uint32_t)((R == 0 ? 4 : 2) + t) << 11);
    const uint32_t b_q = bbase + ((uint32_t)((t & 1) ? 0 : 2) << 11);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float kr = kv[j] * rcp(p[s][j]);  // k e^{E_t - g}
      st_f32(kmaj32_addr(a_hi, cl, j), tf32r(kr * f_hi));
      if (t <= ALO) st_f32(kmaj32_addr(a_lo, cl, j), tf32r(kr * f_lo));
      if (rows) {
        const float f = p[s][j] * f_b;  // e^{g - R_t}
        st_f32(kmaj32_addr(b_q, cl, j), tf32r(qv[j] * f));
        st_f32(kmaj32_addr(b_q + 2048, cl, j), tf32r(kv[j] * f));
      }
    }
  }
}

// T (fp32 64x64) with 16-byte chunks XOR-swizzled by row.
__device__ __forceinline__ int tix(int r, int c) {
  return r * CH + ((((c >> 2) ^ (r & 15)) << 2) | (c & 3));
}

// The off-diagonal blocks of T from its diagonal blocks, by halves.  akk
// holds L transposed (akk[i][r] = L[r][i]); dinv[a][x][rr] = T_aa[rr][x].
// With T1, T2 the inverses of the two 32 x 32 diagonal halves of L and L_C
// its lower-left 32 x 32 block,
//   T1 = [T_00 0; T_10 T_11],  T_10 = -T_11 L_10 T_00  (T_32 likewise),
//   lower-left block of T = -T2 (L_C T1).
// Four phases: P = L_{b+1,b} T_bb and T_{b+1,b} = -T_{b+1,b+1} P for b = 0
// and 2 (P in the unused block (b, b+1) of ti), then X = L_C T1 (block
// (kb, cb) of X in the unused block (cb, kb)), then -T2 X.  A thread owns a
// strip of 4 columns of one row; each phase ends in the body's barrier (sync).
template <class Sync>
__device__ __forceinline__ void solve_offdiag(const float* akk, float* ti, const float* dinv,
                                              int tid, Sync&& sync) {
  if (tid < 128) {
    const int b = 2 * (tid >> 6), a = b + 1, rr = (tid >> 2) & 15, q = tid & 3;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const float l = akk[(16 * b + x) * AKS + 16 * a + rr];
      const float4 t = *reinterpret_cast<const float4*>(ti + tix(16 * b + x, 16 * b + 4 * q));
      acc.x += l * t.x;
      acc.y += l * t.y;
      acc.z += l * t.z;
      acc.w += l * t.w;
    }
    *reinterpret_cast<float4*>(ti + tix(16 * b + rr, 16 * a + 4 * q)) = acc;
  }
  sync();
  if (tid < 128) {
    const int b = 2 * (tid >> 6), a = b + 1, rr = (tid >> 2) & 15, q = tid & 3;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const float d = dinv[(a * 16 + x) * 16 + rr];
      const float4 t = *reinterpret_cast<const float4*>(ti + tix(16 * b + x, 16 * a + 4 * q));
      acc.x += d * t.x;
      acc.y += d * t.y;
      acc.z += d * t.z;
      acc.w += d * t.w;
    }
    *reinterpret_cast<float4*>(ti + tix(16 * a + rr, 16 * b + 4 * q)) =
        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  sync();
  {  // X = L_C T1: rows r in [32, 64), columns of block cb; T1 is zero above its diagonal blocks
    const int cb = tid >> 7, r = 32 + ((tid >> 2) & 31), c0 = 16 * cb + 4 * (tid & 3);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto term = [&](int m) {
      const float l = akk[m * AKS + r];
      const float4 t = *reinterpret_cast<const float4*>(ti + tix(m, c0));
      acc.x += l * t.x;
      acc.y += l * t.y;
      acc.z += l * t.z;
      acc.w += l * t.w;
    };
    if (cb == 0) {  // warp-uniform
#pragma unroll
      for (int m = 0; m < 16; ++m) term(m);
    }
#pragma unroll
    for (int m = 16; m < 32; ++m) term(m);
    *reinterpret_cast<float4*>(ti + tix(16 * cb + (r & 15), 16 * (r >> 4) + (c0 & 15))) = acc;
  }
  sync();
  {  // -T2 X: rows r of block 2 + rb, columns of block cb; T2 is zero above its diagonal blocks
    const int rb = tid >> 7, cb = (tid >> 6) & 1;
    const int r = 32 + 16 * rb + ((tid >> 2) & 15), c0 = 16 * cb + 4 * (tid & 3);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto term = [&](int k) {
      const float t2 = ti[tix(r, k)];
      const float4 x = *reinterpret_cast<const float4*>(ti + tix(16 * cb + (k & 15), 16 * (k >> 4) + 4 * (tid & 3)));
      acc.x += t2 * x.x;
      acc.y += t2 * x.y;
      acc.z += t2 * x.z;
      acc.w += t2 * x.w;
    };
#pragma unroll
    for (int k = 32; k < 48; ++k) term(k);
    if (rb == 1) {  // warp-uniform
#pragma unroll
      for (int k = 48; k < 64; ++k) term(k);
    }
    *reinterpret_cast<float4*>(ti + tix(r, c0)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  sync();
}

// Position pair pidx of the ablation: tile a, row rr and column ii <= rr.
__device__ __forceinline__ void pair_of(int pidx, int& a, int& rr, int& ii) {
  a = pidx / 136;
  const int idx = pidx - 136 * a;
  rr = 0;
  while ((rr + 1) * (rr + 2) / 2 <= idx) ++rr;
  ii = idx - rr * (rr + 1) / 2;
}

// Ablation of the dense diagonal tiles: the four 16x16 diagonal tiles of
// A_qk and A_kk evaluated per position pair in log space,
//   A[r,i] = sum_c q_rc k_ic exp(g_rc - g_ic),   i <= r in the same tile,
// on CUDA cores, which is the evaluation that needs no bound on the decay
// (the orkas.ai page, "Kimi K3 architecture", section "Eine Untergrenze,
// die einen GPU-Codepfad beseitigte", describes the previous generation's
// kernels keeping such a path for the diagonal).  q and k (exact in bf16)
// and g (fp32) are staged as [token][channel] in [0, 64K) of shared memory;
// one thread per position pair walks the channels starting at a
// thread-dependent offset so a warp's loads fall in distinct banks.  Pair
// pidx = tid + 256 n (of 4 x 136) leaves A_qk in aq[n] and A_kk in ak[n].
// Called by all 256 threads of a stage-1 body; sync is its barrier.
template <class Sync>
__device__ __forceinline__ void diagonal_tiles_per_pair(uint8_t* sbp, uint32_t tl, int tid,
                                                        float (&aq)[3], float (&ak)[3], Sync&& sync) {
  uint16_t* sq = reinterpret_cast<uint16_t*>(sbp);
  uint16_t* sk = reinterpret_cast<uint16_t*>(sbp + 16384);
  float* sg = reinterpret_cast<float*>(sbp + 32768);
  const int c = tid & (DP - 1), t_lo = (tid >> 7) * 32;  // this thread: channel c, 32 tokens
#pragma unroll 1
  for (int t0 = t_lo; t0 < t_lo + 32; t0 += 16) {
    float qv[16], kv[16], gv[16];
    tmem_ld16(tl + TA_Q + t0, qv);
    tmem_ld16(tl + TA_K + t0, kv);
    tmem_ld16(tl + TA_G + t0, gv);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      sq[(t0 + j) * DP + c] = __bfloat16_as_ushort(__float2bfloat16_rn(qv[j]));
      sk[(t0 + j) * DP + c] = __bfloat16_as_ushort(__float2bfloat16_rn(kv[j]));
      sg[(t0 + j) * DP + c] = gv[j];
    }
  }
  sync();
#pragma unroll
  for (int n = 0; n < 3; ++n) {
    const int pidx = tid + A_THREADS * n;
    float aqs = 0.f, aks = 0.f;
    if (pidx < 4 * 136) {
      int a, rr, ii;
      pair_of(pidx, a, rr, ii);
      const int r = 16 * a + rr, i = 16 * a + ii;
#pragma unroll 4
      for (int cc = 0; cc < DP; ++cc) {
        const int ch = (cc + tid) & (DP - 1);
        const float e = ex2((sg[r * DP + ch] - sg[i * DP + ch]) * LOG2E);
        const float ki = bf2f(sk[i * DP + ch]) * e;
        aqs = fmaf(bf2f(sq[r * DP + ch]), ki, aqs);
        aks = fmaf(bf2f(sk[r * DP + ch]), ki, aks);
      }
    }
    aq[n] = aqs;
    ak[n] = aks;
  }
  sync();
}

// The fused single-launch prefill (kda_fused_kernel): one CTA per SM, the
// first B * H CTAs walk the state chains and the others run two stage-1
// items at a time, in chunk order, into a ring of R records per chain.
//   ready[c][s]  = j + 1 once the record of chunk j of chain c is complete in
//                  slot s = j % R (stage 1 publishes, the chain waits);
//   consumed[c]  = the chunks of chain c whose records have been copied into
//                  the chain's shared memory (the chain publishes; stage 1
//                  waits before it overwrites a slot);
//   counter      = the next stage-1 item (chunk-major: item w is chunk
//                  w / (B H) of chain w % (B H)).
// All three start at zero.  Each of them, and each chain's ready slots, has
// a 128-byte line of its own (kFlagLine ints apart), so that polls of one
// flag do not slow the stores and polls of the others.  The grid is a
// cooperative launch, so every CTA is resident and a wait on another role
// always ends; each wait is bounded all the same.
constexpr int kFlagLine = 32;  // ints per 128-byte line
struct FusedRing {
  int* ready;     // chain c's slots at ready + c * ready_stride
  int* consumed;  // chain c's at consumed + c * kFlagLine
  int* counter;
  int R, ready_stride;
  // or null: every token's u = beta (v - S'^T k), fp32, [B * T][H][d] like
  // the output (the backward rebuilds its token states from them)
  float* u_out;
};

// Orders this thread's global accesses between the generic proxy (the flags)
// and the async proxy (bulk copies of the records).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int ld_relaxed_gpu(const int* ptr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* ptr, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(int* ptr, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
// Waits until *ptr >= want, for at most two seconds of wall time; `seen` is a
// value of *ptr read earlier (a load issued ahead of need).  Relaxed loads:
// a GPU-scope load reads the coherent copy in L2, and what depends on the
// flag is a bulk copy, issued only once the value has been seen, that reads
// L2 too, where the producer's completed stores were before it published.
// A waiter that can afford latency backs off (sleeps doubling from 256 ns
// to 4 us), which keeps many waiters from crowding the flag's line.
__device__ __forceinline__ bool poll_at_least(const int* ptr, int want, int seen,
                                              bool backoff = false) {
  if (seen >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t ns = backoff ? 256 : 64;
  while (true) {
    if (ld_relaxed_gpu(ptr) >= want) return true;
    if (globaltimer_ns() - t0 > 2000000000ull) return false;
    __nanosleep(ns);
    if (backoff && ns < 4096) ns *= 2;
  }
}
// Named barrier `id` over `n` threads (a part of the CTA).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Stage 1 work list: item w = ((n * seg_len) + (j - j_lo)) * H + h covers
// chunk j of sequence n, head h, for chunks j in [j_lo, j_lo + seg_len).
struct IntraParams {
  const __nv_bfloat16* beta;
  uint8_t* records;
  const int* plan;  // packed sequences: see kda_plan_kernel; null for fixed lengths
  int T, n_seq, H;
  int check_decay;
  int j_lo, seg_len, n_items;
  // fixed lengths in a ring: the record of chunk j of sequence n is
  // n * rec_stride + rec_shift + j (as in StateParams)
  int rec_stride, rec_shift;
  // Overlapped schedule, else null: grid_done[0] counts finished CTAs,
  // grid_done[1] hands out items to a persistent grid.  The CTA that
  // finishes last resets both.
  int* grid_done;
};

// RING: records in a ring (p.rec_stride, p.rec_shift); a separate
// instantiation, so that the others carry none of it.
// The intra-chunk stage run by 256 threads (tid 0..255) over smem_raw: a
// whole CTA of kda_intra_kernel, or one half of a fused CTA (FUSED), whose
// barrier is then the named barrier bar_id over those 256 threads.
template <int DIN, bool PAIRS, bool RING, bool FUSED, typename Params>
__device__ __forceinline__ void intra_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                           const CUtensorMap& tm_g, Params p, const FusedRing& ring,
                                           uint8_t* smem_raw, const int tid, const uint32_t bar_id) {
  // Two CTAs (or CTA halves) per SM loop over (chunk, head) items: taken
  // from a counter (a persistent grid), or without one at a fixed stride
  // over the grid.
  const int warp = tid >> 5;
  auto csync = [&]() {
    if (FUSED)
      named_sync(bar_id, A_THREADS);
    else
      __syncthreads();
  };
  const int c = tid & (DP - 1), hh = tid >> 7;  // key channel (TMEM lane); token half
  const int ta[2] = {hh ? 1 : 0, hh ? 2 : 3};   // the token tiles this thread owns
  const int H = p.H;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sbp = smem_raw + (sb - raw);
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sbp + A_MISC);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sbp + A_MISC + 16);
  int* s_abort = reinterpret_cast<int*>(sbp + A_MISC + 20);
  int* s_pub = reinterpret_cast<int*>(sbp + A_MISC + 32);  // fused: {chain, chunk} to publish
  float* s_beta = reinterpret_cast<float*>(sbp + A_MISC + 64);    // [64]
  float* s_gamma = reinterpret_cast<float*>(sbp + A_MISC + 512);  // [128], 16-byte aligned

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
    *s_abort = 0;
    s_pub[1] = -1;
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_s, TA_COLS);
    if (!FUSED) tmem_relinquish();  // (a fused CTA has a second allocation to make)
  }
  tc_fence_before_sync();
  csync();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_base_s;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  uint32_t tma_phase = 0, mma_phase = 0;
  bool ok = true;

  auto wait_all = [&](uint64_t* bar, uint32_t& phase) -> bool {
    if (!mbar_wait(bar, phase)) {
      *s_abort = 1;
      set_status(6);
    }
    phase ^= 1u;
    csync();
    tc_fence_after_sync();
    return *s_abort == 0;
  };
  auto operands_ready = [&]() {
    fence_proxy_async_smem();
    tc_fence_before_sync();
    csync();
    tc_fence_after_sync();
  };

  // item w -> head, first token, valid tokens and record index (valid <= 0:
  // past the end of a packed sequence)
  struct Item {
    int h, t0, valid, qrec, chain, chunk;
  };
  auto item_of = [&](int w) {
    Item it{};
    it.h = w % H;
    const int item_r = w / H;
    int n = item_r / p.seg_len, jc = p.j_lo + item_r % p.seg_len;
    if (FUSED) {  // chunk-major: all chains of chunk j before chunk j + 1
      it.chain = w % (p.n_seq * H);
      n = it.chain / H;
      jc = w / (p.n_seq * H);
    }
    it.chunk = jc;
    int seq0, len;
    if (FUSED) {
      seq0 = n * p.T;
      len = p.T;
      it.qrec = n * ring.R + jc % ring.R;
    } else if (p.plan) {
      seq0 = p.plan[p.n_seq + 1 + n];
      len = p.plan[2 * p.n_seq + 1 + n];
      it.qrec = p.plan[n] + jc;
    } else {
      seq0 = n * p.T;
      len = p.T;
      it.qrec = RING ? n * p.rec_stride + p.rec_shift + jc : n * ((p.T + CH - 1) / CH) + jc;
    }
    it.t0 = seq0 + CH * jc;
    it.valid = min(CH, len - CH * jc);
    return it;
  };
  int* s_item = reinterpret_cast<int*>(sbp + A_MISC + 24);
  // next item: from the shared counter (thread 0 takes a ticket with claim()
  // some time before next_item needs it, so the atomic's round trip overlaps
  // work), else a fixed stride over the grid.  The first barrier keeps the
  // write behind every read of the previous value (an empty item skips the
  // body's barriers).
  int* const counter = FUSED ? ring.counter : p.grid_done ? p.grid_done + 1 : nullptr;
  auto claim = [&]() -> int { return tid == 0 && counter ? atomicAdd(counter, 1) : 0; };
  auto next_item = [&](int w, int ticket) -> int {
    if (!counter) return w + gridDim.x;
    csync();
    if (tid == 0) *s_item = ticket;
    csync();
    return *s_item;
  };
  // The inputs of item w: thread 0 issues the TMA loads of its q, k and log
  // alpha tiles, threads below its length load its beta.  Called by all
  // threads; returns whether loads were issued (the same on every thread).
  // Each item's loads are issued while the item before it finishes, into
  // space that item no longer uses.
  auto prefetch = [&](int w, float& beta_reg) -> bool {
    beta_reg = 0.f;
    if (w >= p.n_items) return false;
    const Item it = item_of(w);
    if (it.valid <= 0) return false;
    if (tid < it.valid) beta_reg = __bfloat162float(p.beta[(size_t)(it.t0 + tid) * H + it.h]);
    if (tid == 0) {
      mbar_arrive_expect_tx(bar_tma, 3u * (DIN / 64) * 8192u);
#pragma unroll
      for (int b = 0; b < DIN / 64; ++b) {
        tma_load_3d(sbp + A_RQ + b * 8192, &tm_q, bar_tma, b * 64, it.h, it.t0);
        tma_load_3d(sbp + A_RK + b * 8192, &tm_k, bar_tma, b * 64, it.h, it.t0);
        tma_load_3d(sbp + A_RG + b * A_RG_LBO, &tm_g, bar_tma, b * 64, it.h, it.t0);
      }
    }
    return true;
  };
  int w = next_item(counter ? 0 : (int)blockIdx.x - (int)gridDim.x, claim());
  // Fused: thread 0 publishes a record once its bulk stores have completed,
  // some time after it issued them (the wait then costs nothing), and while
  // the next item's first product runs (which hides part of the release).
  // The bytes and the flag reach L2 by different paths, so the flag is a
  // release at GPU scope: a chain that sees it finds the bytes there.  Every
  // record is published before its body can wait for a ring slot, so no
  // record waits behind another chain's progress.  (Publishing two records
  // per release, or from another thread after a barrier, measured slower.)
  auto publish = [&]() {  // thread 0
    bulk_wait_all();
    fence_proxy_async_global();
    if (s_pub[1] >= 0) {
      st_release_gpu(ring.ready + s_pub[0] * ring.ready_stride + s_pub[1] % ring.R, s_pub[1] + 1);
      s_pub[1] = -1;
    }
  };
  float beta_t;
  bool pending = prefetch(w, beta_t);
  while (ok && w < p.n_items) {
  const Item cur = item_of(w);
  if (cur.valid <= 0) {
    w = next_item(w, claim());
    pending = prefetch(w, beta_t);
    continue;
  }
  const int h = cur.h, valid = cur.valid, qrec = cur.qrec;
  // fused: the chain's progress as of now, read ahead of the first store
  const int consumed_seen =
      FUSED && tid == 0 ? ld_relaxed_gpu(ring.consumed + cur.chain * kFlagLine) : 0;
  uint8_t* rec = p.records + ((size_t)qrec * H + h) * REC_BYTES;
  int w_next = p.n_items;
  float beta_next = 0.f;
  bool pending_next = false;

  if (DIN == 64) {  // upper channel half of the raw tiles stays zero
    for (uint32_t off = tid * 16; off < 8192; off += A_THREADS * 16) {
      st_shared_v4(sb + A_RQ + 8192 + off, 0, 0, 0, 0);
      st_shared_v4(sb + A_RK + 8192 + off, 0, 0, 0, 0);
      st_shared_v4(sb + A_RG1 + off, 0, 0, 0, 0);
    }
  }
  // L[r][i] = (i <= r), I[r][i] = (i == r), both restricted to valid tokens i
  const OperandLayout LM = kmajor(sb + A_LM, 0), IM = kmajor(sb + A_IM, 0);
  {
    const int r = tid >> 2, i_lo = (tid & 3) * 16;
#pragma unroll
    for (int i0 = i_lo; i0 < i_lo + 16; i0 += 8) {
      float l[8], e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + j;
        l[j] = (i <= r && i < valid) ? 1.f : 0.f;
        e[j] = (i == r && i < valid) ? 1.f : 0.f;
      }
      st8(layout_addr(LM, r, i0), l);
      st8(layout_addr(IM, r, i0), e);
    }
  }
  if (tid < CH) s_beta[tid] = beta_t;
  fence_proxy_async_smem();
  tc_fence_before_sync();
  csync();
  tc_fence_after_sync();

  ok = wait_all(bar_tma, tma_phase);
  if (ok && p.check_decay) {
    bool bad = false;
    const OperandLayout RG = kmajor(sb + A_RG, A_RG_LBO);
    for (int i = 32 * hh; i < valid && i < 32 * hh + 32; ++i) {
      const float la = bf2f(ld_shared_u16(layout_addr(RG, i, c)));
      bad |= !(la >= -5.f && la <= 0.f);
    }
    if (bad) set_status(5);
  }
  constexpr uint32_t ID_T = make_idesc(128, 64, true, false);  // bf16, A MN-major
  if (ok && tid == 0) {
    const uint64_t dq = layout_desc(mnmajor(sb + A_RQ, 8192), 0, 0);
    const uint64_t dk = layout_desc(mnmajor(sb + A_RK, 8192), 0, 0);
    const uint64_t dg = layout_desc(mnmajor(sb + A_RG, A_RG_LBO), 0, 0);
    const uint64_t dl = layout_desc(LM, 0, 0), di = layout_desc(IM, 0, 0);
#pragma unroll
    for (int k0 = 0; k0 < CH; k0 += 16) {
      const uint64_t bl = desc_adv(dl, k0, false), bi = desc_adv(di, k0, false);
      umma_bf16(tmem + TA_G, desc_adv(dg, k0, true), bl, ID_T, k0 > 0);
      umma_bf16(tmem + TA_Q, desc_adv(dq, k0, true), bi, ID_T, k0 > 0);
      umma_bf16(tmem + TA_K, desc_adv(dk, k0, true), bi, ID_T, k0 > 0);
    }
    umma_commit(bar_mma);
  }
  if (ok) ok = wait_all(bar_mma, mma_phase);

  // ---- decay factors of this thread's channel and tiles: E[b] = g at the
  // end of tile b; p[s][j] = e^{g - E} of token 16 ta[s] + j, in [1, e^80]
  float E[4], Eo[2], Ep[2], pr[2][16];
  if (ok) {
#pragma unroll
    for (int b = 0; b < 4; ++b) E[b] = tmem_ld1(tl + TA_G + 16 * b + 15);
    float g0[16], g1[16];
    tmem_ld16(tl + TA_G + 16 * ta[0], g0);
    tmem_ld16(tl + TA_G + 16 * ta[1], g1);
    tmem_ld_wait();
    Eo[0] = hh ? E[1] : E[0];
    Eo[1] = hh ? E[2] : E[3];
    Ep[0] = hh ? E[0] : 0.f;
    Ep[1] = hh ? E[1] : E[2];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      pr[0][j] = ex2((g0[j] - Eo[0]) * LOG2E);
      pr[1][j] = ex2((g1[j] - Eo[1]) * LOG2E);
    }
  }

  // the previous item's last stores read [56K, 64K) and [81K, 97K), which the
  // M1 operands (and the ablation's staging) below overwrite
  if (tid == 0) bulk_wait_reads();
  csync();
  // ablation only: the diagonal tiles per position pair, while g is in TMEM
  float pq[3], pk[3];
  if (PAIRS && ok) diagonal_tiles_per_pair(sbp, tl, tid, pq, pk, csync);

  // ---- M1 in two passes of one kind::tf32 product each, K-major fp32
  // operands: A = key rows under the references of two row tiles
  // ([128 keys][128 channels]), B = those tiles' token rows ([64][128]).
  // Pass 0 writes TMEM columns TA_A, pass 1 TA_G (g is no longer needed).
  OperandLayout XA = kmajor(sb + A_XH, 16384), KBA = kmajor(sb + A_KBH, 8192);
  XA.esize = 4;
  KBA.esize = 4;
  constexpr uint32_t ID_M1 = make_idesc_tf32(128, 64, false, false);
  const uint32_t cl = (uint32_t)(c & 31) * 4;
  const uint32_t abase = sb + A_XH + (uint32_t)(c >> 5) * 16384;
  const uint32_t bbase = sb + A_KBH + (uint32_t)(c >> 5) * 8192;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    if (!ok) break;
    if (pass == 0) build_m1_pass<0>(abase, bbase, cl, tl, pr, E, Eo, Ep, ta);
    if (pass == 1) build_m1_pass<1>(abase, bbase, cl, tl, pr, E, Eo, Ep, ta);
    operands_ready();
    if (tid == 0) {
      const uint32_t d = tmem + (pass == 0 ? TA_A : TA_G);
#pragma unroll
      for (int k0 = 0; k0 < DP; k0 += 8)
        umma_tf32(d, layout_desc(XA, 0, k0), layout_desc(KBA, 0, k0), ID_M1, k0 > 0);
      umma_commit(bar_mma);
      if (FUSED && pass == 0) publish();  // the previous item's record
    }
    ok = wait_all(bar_mma, mma_phase);
  }

  float* akk = reinterpret_cast<float*>(sbp + A_AKK);
  float* ti = reinterpret_cast<float*>(sbp + A_TI);
  const OperandLayout AQ = mnmajor(sb + A_STG + REC_AQ, 8192);
  const OperandLayout QT = mnmajor(sb + A_STG + REC_QT, 16384);
  const OperandLayout KBAR = kmajor(sb + A_STG + REC_KBAR, 0);
  const OperandLayout KT = kmajor(sb + A_KT, 0);
  const OperandLayout TB = kmajor(sb + A_STG + REC_TB, 0);
  const OperandLayout WT = mnmajor(sb + A_WST, 16384);
  if (ok) {
    // ---- A_qk (fp16 record image, MN-major: N = r, K = i) and beta-scaled
    // strictly-lower A_kk (fp32, stored transposed, akk[i * AKS + r] =
    // L[r][i]: the solve reads L by columns).  TMEM lane = key: pass 0 (TA_A)
    // lanes 0..63 are the keys of row tile 3 and lanes 64..111 keys 0..47 of
    // row tile 2; pass 1 (TA_G) lanes 0..31 keys of row tile 1 and lanes
    // 32..47 keys 0..15 of row tile 0.  Columns: q then k rows of the odd
    // tile, then of the even one.  hh = 0 takes the q columns (A_qk), hh = 1
    // the k columns (A_kk).
    auto extract = [&](uint32_t cols, int a, int i) {
      float v[16];
      tmem_ld16(tl + cols + ((a & 1) ? 0 : 32) + 16 * hh, v);
      tmem_ld_wait();
      if (i >= 16 * (a + 1)) return;  // a key after the row tile
      if (hh == 0) {
#pragma unroll
        for (int h8 = 0; h8 < 16; h8 += 8) {
          float x[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) x[j] = i <= 16 * a + h8 + j ? v[h8 + j] : 0.f;
          st8h(layout_addr(AQ, 16 * a + h8, i), x);
        }
      } else {
#pragma unroll
        for (int q4 = 0; q4 < 16; q4 += 4) {
          const int r0 = 16 * a + q4;
          float4 x;
          x.x = i < r0 ? s_beta[r0] * v[q4] : 0.f;
          x.y = i < r0 + 1 ? s_beta[r0 + 1] * v[q4 + 1] : 0.f;
          x.z = i < r0 + 2 ? s_beta[r0 + 2] * v[q4 + 2] : 0.f;
          x.w = i < r0 + 3 ? s_beta[r0 + 3] * v[q4 + 3] : 0.f;
          *reinterpret_cast<float4*>(akk + i * AKS + r0) = x;
        }
      }
    };
    const int quad = c >> 5;  // warp-uniform
    extract(TA_A, quad < 2 ? 3 : 2, c & 63);
    if (quad < 2) extract(TA_G, quad == 0 ? 1 : 0, c & 31);
    if (hh == 0 && c < CH) {  // A_qk is zero above the diagonal tiles
      const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int r0 = 0; r0 < 16 * (c >> 4); r0 += 8) st8h(layout_addr(AQ, r0, c), z);
    }
    if (PAIRS) {  // the ablation's diagonal tiles replace the dense ones
      csync();
#pragma unroll
      for (int n = 0; n < 3; ++n) {
        const int pidx = tid + A_THREADS * n;
        if (pidx < 4 * 136) {
          int a, rr, ii;
          pair_of(pidx, a, rr, ii);
          const int r = 16 * a + rr, i = 16 * a + ii;
          *reinterpret_cast<__half*>(sbp + (layout_addr(AQ, r, i) - sb)) = __float2half_rn(pq[n]);
          if (ii < rr) akk[i * AKS + r] = s_beta[r] * pk[n];
        }
      }
    }
    // ---- (k e^g)^T (bf16, M2 operand), q e^g and k e^{g_C - g} (fp16 record
    // images), for this thread's channel and tiles
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const int a = ta[s2];
      float qv[16], kv[16];
      tmem_ld16(tl + TA_Q + 16 * a, qv);
      tmem_ld16(tl + TA_K + 16 * a, kv);
      tmem_ld_wait();
      const float ge = ex2(Eo[s2] * LOG2E);             // e^{E_a}
      const float f3 = ex2((E[3] - Eo[s2]) * LOG2E);   // e^{E_3 - E_a}
#pragma unroll
      for (int h8 = 0; h8 < 16; h8 += 8) {
        float kt[8], qt[8], kb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float pj = pr[s2][h8 + j];
          const float gam = pj * ge;  // e^{g_i}
          kt[j] = kv[h8 + j] * gam;
          qt[j] = qv[h8 + j] * gam;
          kb[j] = kv[h8 + j] * rcp(pj) * f3;  // e^{g_C - g_i}
        }
        const int i0 = 16 * a + h8;
        st8(layout_addr(KT, c, i0), kt);
        st8h(layout_addr(QT, i0, c), qt);
        st8h(layout_addr(KBAR, c, i0), kb);
      }
    }
    if (hh == 0) s_gamma[c] = ex2(E[3] * LOG2E);
    fence_proxy_async_smem();
    csync();
    if (tid == 0) {  // q e^g, K-bar and A_qk are final: store them while the solve runs
      // fused: the slot's previous record (chunk - R) must have been copied in
      const int need = cur.chunk - ring.R + 1;
      const bool slot_free = !FUSED || poll_at_least(ring.consumed + cur.chain * kFlagLine, need,
                                                     consumed_seen, true);
      if (slot_free) {
        if (FUSED) fence_proxy_async_global();
        bulk_s2g(rec + REC_QT, sb + A_STG + REC_QT, REC_TB - REC_QT);
        bulk_commit();
      } else {
        *s_abort = 1;
        set_status(6);
      }
    }
    // the ticket for the item after this one, read once the solve is done
    const int ticket = claim();

    // ---- T = (I + A_kk)^-1, unit lower triangular, in fp32.  L = I + A_kk is
    // read transposed (akk[i][r] = L[r][i]); T lives in ti with its 16-byte
    // chunks XOR-swizzled by row, so row-wise float4 traffic is conflict-free.
    float* dinv = reinterpret_cast<float*>(sbp + A_DINV);  // [4][16][16], dinv[a][x][rr] = T_aa[rr][x]
    // diagonal blocks by forward substitution: thread (a, j) solves column j of block a
    if (tid < 64) {
      const int a = tid >> 4, j = tid & 15;
      float x[16];
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) x[rr] = rr == j ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < 15; ++m) {
        const float xm = x[m];
#pragma unroll
        for (int rr = m + 1; rr < 16; ++rr) x[rr] -= akk[(16 * a + m) * AKS + 16 * a + rr] * xm;
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) ti[tix(16 * a + rr, 16 * a + j)] = x[rr];
      float4* drow = reinterpret_cast<float4*>(dinv + (a * 16 + j) * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) drow[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
    csync();
    // off-diagonal blocks: T_10 and T_32, then the lower-left 32 x 32 block
    solve_offdiag(akk, ti, dinv, tid, csync);
    // the next item's inputs land where this item's first record stores read
    // (and in A_RG1): once those reads are done, issue them
    w_next = next_item(w, ticket);
    if (tid == 0) bulk_wait_reads();
    pending_next = prefetch(w_next, beta_next);
    // ---- T diag(beta) in bf16 (rows r, K = i), lower triangle only
    {
      const int r = tid >> 2, i_lo = (tid & 3) * 16;
#pragma unroll
      for (int i0 = i_lo; i0 < i_lo + 16; i0 += 8) {
        const float4 t0 = *reinterpret_cast<const float4*>(ti + tix(r, i0));
        const float4 t1 = *reinterpret_cast<const float4*>(ti + tix(r, i0 + 4));
        const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j;
          x[j] = i <= r ? tv[j] * s_beta[i] : 0.f;
        }
        st8(layout_addr(TB, r, i0), x);
      }
    }
    operands_ready();
    if (tid == 0) {
      constexpr uint32_t ID_W = make_idesc(128, 64, false, false);
      const uint64_t dkt = layout_desc(KT, 0, 0), dtb = layout_desc(TB, 0, 0);
#pragma unroll
      for (int k0 = 0; k0 < CH; k0 += 16)
        umma_bf16(tmem + TA_W, desc_adv(dkt, k0, false), desc_adv(dtb, k0, false), ID_W, k0 > 0);
      umma_commit(bar_mma);
    }
    ok = wait_all(bar_mma, mma_phase);
  }
  if (ok) {
    // ---- W (fp16, N = r, K = c) from W^T in TMEM (lane = c), into the (k e^g)^T slot
    float w0[16], w1[16];
    tmem_ld16(tl + TA_W + 32 * hh, w0);
    tmem_ld16(tl + TA_W + 32 * hh + 16, w1);
    tmem_ld_wait();
    st8h(layout_addr(WT, 32 * hh, c), w0);
    st8h(layout_addr(WT, 32 * hh + 8, c), w0 + 8);
    st8h(layout_addr(WT, 32 * hh + 16, c), w1);
    st8h(layout_addr(WT, 32 * hh + 24, c), w1 + 8);
    fence_proxy_async_smem();
    csync();
    if (tid == 0) {
      bulk_s2g(rec + REC_WT, sb + A_WST, REC_QT - REC_WT);
      bulk_s2g(rec + REC_TB, sb + A_STG + REC_TB, REC_G - REC_TB);
      bulk_s2g(rec + REC_G, smem_u32(s_gamma), 512);
      bulk_commit();
      if (FUSED) {
        s_pub[0] = cur.chain;
        s_pub[1] = cur.chunk;
      }
    }
  }
  w = w_next;
  beta_t = beta_next;
  pending = pending_next;
  }  // items
  // loads still in flight after a failed wait land before the CTA's memory goes away
  if (pending && tid == 0) mbar_wait(bar_tma, tma_phase);
  if (tid == 0) {
    if (FUSED)
      publish();  // the last record
    else
      bulk_wait_all();
  }
  tc_fence_before_sync();
  csync();
  if (warp == 0) tmem_dealloc(tmem, TA_COLS);
  if (!FUSED && p.grid_done && tid == 0) {
    // This grid was allowed to start before the previous segment's state
    // pass finished.  The CTA that finishes last waits for that grid, so
    // this grid completes only after it: the next state pass, which reads
    // the state it carried, is ordered after both.
    const int ticket = atomicAdd(p.grid_done, 1);
    if (ticket == (int)(gridDim.x * gridDim.y) - 1) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      p.grid_done[0] = 0;
      p.grid_done[1] = 0;
    }
  }
}

template <int DIN, bool PAIRS, bool RING = false>
__global__ void __launch_bounds__(A_THREADS, 2)
    kda_intra_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_g, IntraParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  intra_body<DIN, PAIRS, RING, false, const IntraParams>(tm_q, tm_k, tm_g, p, FusedRing{}, smem_raw,
                                                        threadIdx.x, 0);
}

// Stage 2 covers chunks [j_lo, j_hi) of every sequence.  The state entering
// chunk j_lo is s0 when j_lo == 0, else the carried state; the state after a
// sequence's last chunk goes to s1, else (the range ends earlier) to carry.
struct StateParams {
  const uint8_t* records;
  const float* s0;
  float* s1;
  float* carry;  // [n_seq][H][128][128] fp32, or null for a single range
  void* out;
  const int* plan;  // packed sequences: see kda_plan_kernel; null for fixed lengths
  int T, n_seq, H;
  int j_lo, j_hi;
  float scale;
  float* ckpt;  // state after every ckpt_every chunks ([n_seq][n_ckpt][H][d][d]), or null
  int ckpt_every, n_ckpt;
  // Segment scan (segs > 1): the n_seq sequences of this launch are segments
  // of segs each of n_seq / segs real sequences (segment p of sequence b is
  // sequence b * segs + p).  phase 1 walks every segment: segment 0 from the
  // real initial state with outputs, later segments twice, as the plane
  // blockIdx.z = 0 from a zero state (their zero-start state Z) and
  // blockIdx.z = 1 from the identity with no values (their transition M),
  // both without outputs; every walk leaves its last state in its plane of
  // carry.  phase 2 walks segments 1.. again with outputs from the entry
  // states the scan left in carry plane 0, the last one into s1.
  int segs, phase;
  // fixed lengths: the record of chunk j of sequence n is
  // n * rec_stride + rec_shift + j (one record per chunk, or a ring of two
  // segments; set by the host per launch)
  int rec_stride, rec_shift;  // read by the RING instantiation only
};

// Stage 2 warp roles: warps 0-7 run the elementwise part of the serial
// chain (two per TMEM lane quadrant, splitting columns); warps 8-11 drain
// finished output tiles from TMEM to global memory, double-buffered; warp 12
// (one lane) issues every MMA and every load.  Issuing is kept off the chain
// warps because an issuing thread stalls while the tensor core's queue is
// full.  Hand-offs are mbarriers (bounded waits), never named barriers, so
// a timeout anywhere unwinds every role.
// Largest |state| or |u| entry the fp16 operands of the state pass carry
// (fp16 max 65504); a larger or non-finite entry sets KDA_ERR_RANGE.
constexpr float kOperandMax = 60000.f;
constexpr int B_CHAIN = 256;
constexpr int B_OUTPUT = 128;
constexpr int B_THREADS = B_CHAIN + B_OUTPUT + 32;

// SCAN: the walks of a segment scan (p.phase 1 or 2); RING: records in a
// ring (p.rec_stride, p.rec_shift).  The plain pass is a separate
// instantiation so that it carries none of that logic.
// A CTA of the fused launch (see FusedRing) runs either one state chain (its
// first B_THREADS threads) or two stage-1 bodies.
constexpr int F_THREADS = 2 * A_THREADS;
constexpr uint32_t F_SMEM = 2 * A_SMEM > B_SMEM ? 2 * A_SMEM : B_SMEM;
static_assert(F_THREADS >= B_THREADS, "the state pass fits a fused CTA");

template <int DIN, typename OutT, bool SCAN, bool RING = false>
__global__ void __launch_bounds__(B_THREADS, 1)
    kda_state_kernel(const __grid_constant__ CUtensorMap tm_v, StateParams p) {
  // Every CTA of this grid holds its SM from here on: the next segment's
  // intra-chunk stage (a programmatic dependent) may start on the other SMs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int half = (warp >> 2) & 1;           // chain warps: which half of the columns
  const int v = 32 * (warp & 3) + (tid & 31);  // TMEM lane = value channel
  const int h = blockIdx.x, n = blockIdx.y, H = p.H;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sbp = smem_raw + (sb - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sbp + B_MISC);  // [2] record + v tile landed
  uint64_t* mma_a = full + 2;     // D = -S^T [W; q e^g]^T done
  uint64_t* mma_b = full + 3;     // S update and the rest of O done
  uint64_t* o_full = full + 4;    // [2] output tile ready
  uint64_t* o_empty = full + 6;   // [2] output tile drained
  uint64_t* st_ready = full + 8;  // chain -> issuer: S^T operand written
  uint64_t* ut_ready = full + 9;  // chain -> issuer: U^T operand written, state decayed
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sbp + B_MISC + 96);
  int* s_abort = reinterpret_cast<int*>(sbp + B_MISC + 100);
  int* s_range = reinterpret_cast<int*>(sbp + B_MISC + 104);

  int tok0, len, base;
  if (p.plan) {
    tok0 = p.plan[p.n_seq + 1 + n];
    len = p.plan[2 * p.n_seq + 1 + n];
    base = p.plan[n];
  } else {
    tok0 = n * p.T;
    len = p.T;
    base = RING ? n * p.rec_stride + p.rec_shift : n * ((p.T + CH - 1) / CH);
  }
  const int nch_seq = len > 0 ? (len + CH - 1) / CH : 0;
  const int jb = p.j_lo, nchunks = max(0, min(p.j_hi, nch_seq) - jb);  // j below is jb + local
  const size_t sbase = (size_t)(n * H + h) * DIN * DIN;
  // the walk this CTA does: kind 0 the plain recurrence with outputs, 1 the
  // transition (identity start, no values, no outputs), 2 the zero-start
  // state (no outputs); and where its first state comes from and its last
  // state goes
  const int seg = SCAN ? n % p.segs : 0;
  const size_t real = (size_t)((SCAN ? n / p.segs : n) * H + h) * DIN * DIN;
  const size_t plane = (size_t)p.n_seq * H * DIN * DIN;
  float* carry = p.carry ? p.carry + (SCAN ? blockIdx.z * plane : 0) + sbase : nullptr;
  int kind = 0;
  if (SCAN && p.phase == 1 && seg > 0) kind = blockIdx.z ? 1 : 2;
  if (SCAN && ((p.phase == 1 && seg == 0 && blockIdx.z) || (p.phase == 2 && seg == 0))) return;
  const bool last_range = jb + nchunks == nch_seq;
  const float* s_in;
  float* s_out;
  if (!SCAN) {
    s_in = jb == 0 ? (p.s0 ? p.s0 + sbase : nullptr) : carry;
    s_out = last_range ? (p.s1 ? p.s1 + sbase : nullptr) : carry;
  } else if (p.phase == 1) {
    s_in = jb > 0 ? carry : (kind == 0 && p.s0 ? p.s0 + real : nullptr);
    s_out = carry;
  } else {
    s_in = carry;
    s_out = last_range && seg == p.segs - 1 && p.s1 ? p.s1 + real : nullptr;
  }
  const bool ident = SCAN && kind == 1 && jb == 0;  // the transition walk starts from I
  const bool outputs = !SCAN || kind == 0;
  if (nchunks == 0) {  // nothing in this range; a sequence with no tokens keeps its state
    if (jb == 0 && nch_seq == 0 && s_out)
      for (int i = threadIdx.x; i < DIN * DIN; i += blockDim.x)
        s_out[i] = ident ? (i / DIN == i % DIN ? 1.f : 0.f) : (s_in ? s_in[i] : 0.f);
    return;
  }
  constexpr uint32_t kVBytes = (DIN / 64) * 8192u;
  auto issue_loads = [&](int j, int buf) {
    const uint8_t* rec = p.records + ((size_t)(base + jb + j) * H + h) * REC_BYTES;
    uint8_t* dst = sbp + (buf ? B_REC1 : B_REC0);
    uint8_t* vdst = sbp + (buf ? B_V1 : B_V0);
    mbar_arrive_expect_tx(&full[buf], REC_LOAD + (SCAN && kind == 1 ? 0u : kVBytes));
    bulk_g2s(dst, rec, REC_LOAD, &full[buf]);
    if (!SCAN || kind != 1) {
#pragma unroll
      for (int b = 0; b < DIN / 64; ++b)
        tma_load_3d(vdst + b * 8192, &tm_v, &full[buf], b * 64, h, tok0 + CH * (jb + j));
    }
  };
  auto gamma_of = [&](int buf) {
    return reinterpret_cast<const float*>(sbp + (buf ? B_REC1 : B_REC0) + REC_G);
  };

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(mma_a, 1);
    mbar_init(mma_b, 1);
    mbar_init(&o_full[0], 1);
    mbar_init(&o_full[1], 1);
    mbar_init(&o_empty[0], B_OUTPUT);
    mbar_init(&o_empty[1], B_OUTPUT);
    mbar_init(st_ready, B_CHAIN);
    mbar_init(ut_ready, B_CHAIN);
    mbar_fence_init();
    *s_abort = 0;
    *s_range = 0;
    if (nchunks > 0) issue_loads(0, 0);
    if (nchunks > 1) issue_loads(1, 1);
  }
  if (DIN == 64) {
    for (uint32_t off = tid * 16; off < 8192; off += B_THREADS * 16) {
      st_shared_v4(sb + B_V0 + 8192 + off, 0, 0, 0, 0);
      st_shared_v4(sb + B_V1 + 8192 + off, 0, 0, 0, 0);
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_s, TB_COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_base_s;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const OperandLayout ST = kmajor(sb + B_ST, 16384);  // M = v, K = c
  const OperandLayout UT = kmajor(sb + B_UT, 0);      // M = v, K = i
  auto fail = [&]() {
    *s_abort = 1;
    set_status(6);
  };

  if (warp == B_THREADS / 32 - 1) {
    // ---------------- issuer: one lane issues every MMA and every load
    if ((tid & 31) == 0 && nchunks > 0) {
      constexpr uint32_t ID_V = make_idesc(128, 64, true, false);                 // bf16
      constexpr uint32_t ID_O2 = make_idesc(128, 64, false, true, true, true);    // fp16, -A
      constexpr uint32_t ID_S = make_idesc(128, 128, false, false, false, true);  // fp16
      // M3 of chunk j, U~^T = V^T (T diag beta)^T, needs no state: it is
      // issued as soon as record j lands, ahead of the chain's own products.
      auto issue_m3 = [&](int j) {
        if (SCAN && kind == 1) return;  // no values: U~ = 0
        const int b = j & 1;
        const uint32_t rb = sb + (b ? B_REC1 : B_REC0), vb = sb + (b ? B_V1 : B_V0);
        const uint64_t dva = layout_desc(mnmajor(vb, 8192), 0, 0);
        const uint64_t dtb = layout_desc(kmajor(rb + REC_TB, 0), 0, 0);
#pragma unroll
        for (int k0 = 0; k0 < CH; k0 += 16)
          umma_bf16(tmem + TB_UT + 64 * b, desc_adv(dva, k0, true), desc_adv(dtb, k0, false),
                    ID_V, k0 > 0);
      };
      int issued = min(nchunks, 2), landed = 0;  // record loads issued / seen complete
      bool ok = mbar_wait(&full[0], 0);
      if (ok) {
        landed = 1;
        tc_fence_after_sync();
        issue_m3(0);
      }
      for (int j = 0; j < nchunks && ok; ++j) {
        const int buf = j & 1, ob = j & 1;
        const uint32_t rb = sb + (buf ? B_REC1 : B_REC0);
        const uint32_t td = tmem + TB_D + 128 * ob;
        if (!(ok = mbar_wait(st_ready, j & 1))) break;
        if (j >= 2 && !(ok = mbar_wait(&o_empty[ob], ((j - 2) >> 1) & 1))) break;
        tc_fence_after_sync();
        {  // M4, D = -S^T W^T, alone (N = 64): the chain waits only for it.  The
           // first half of M5, -S^T (q e^g)^T, follows into the next 64 columns
           // and runs while the chain forms U^T.
          const uint64_t dst = layout_desc(ST, 0, 0);
          const uint64_t dw = layout_desc(mnmajor(rb + REC_WT, 16384), 0, 0);
          const uint64_t dq = layout_desc(mnmajor(rb + REC_QT, 16384), 0, 0);
#pragma unroll
          for (int k0 = 0; k0 < DP; k0 += 16)
            umma_bf16(td, desc_adv(dst, k0, false, 16384), desc_adv(dw, k0, true), ID_O2, k0 > 0);
          umma_commit(mma_a);
#pragma unroll
          for (int k0 = 0; k0 < DP; k0 += 16)
            umma_bf16(td + 64, desc_adv(dst, k0, false, 16384), desc_adv(dq, k0, true), ID_O2,
                      k0 > 0);
        }
        if (!(ok = mbar_wait(ut_ready, j & 1))) break;
        tc_fence_after_sync();
        {
          const uint64_t dut = layout_desc(UT, 0, 0);
          const uint64_t daq = layout_desc(mnmajor(rb + REC_AQ, 8192), 0, 0);
          const uint64_t dkb = layout_desc(kmajor(rb + REC_KBAR, 0), 0, 0);
          // M6 first: the chain waits only for the state update; the second
          // half of M5 (the output) runs while the chain rebuilds S^T
#pragma unroll
          for (int k0 = 0; k0 < CH; k0 += 16)
            umma_bf16(tmem + TB_S, desc_adv(dut, k0, false), desc_adv(dkb, k0, false), ID_S, 1);
          umma_commit(mma_b);
#pragma unroll
          for (int k0 = 0; k0 < CH; k0 += 16)
            umma_bf16(td + 64, desc_adv(dut, k0, false), desc_adv(daq, k0, true), ID_O2, 1);
          umma_commit(&o_full[ob]);
        }
        if (j + 2 < nchunks) {  // buffer buf is consumed once every product of chunk j is done
          if (!(ok = mbar_wait(&o_full[ob], (j >> 1) & 1))) break;
          fence_proxy_async_smem();
          issue_loads(j + 2, buf);
          ++issued;
        }
        if (j + 1 < nchunks) {
          if (!(ok = mbar_wait(&full[buf ^ 1], ((j + 1) >> 1) & 1))) break;
          ++landed;
          tc_fence_after_sync();
          issue_m3(j + 1);
        }
      }
      if (!ok) {
        fail();
        // let copies already issued land before the CTA's memory goes away
        for (int r = landed; r < issued; ++r) mbar_wait(&full[r & 1], (r >> 1) & 1, 100000000ull);
      }
    }
  } else if (warp >= B_CHAIN / 32) {
    // ---------------- output warps: thread = value channel v, all 64 tokens
    for (int j = 0; j < nchunks; ++j) {
      const int ob = j & 1;
      if (!mbar_wait(&o_full[ob], (j >> 1) & 1)) {
        fail();
        break;
      }
      tc_fence_after_sync();
      const int valid = min(CH, len - CH * (jb + j));
      float o[64];
      tmem_ld64(tl + TB_D + 128 * ob + 64, o);  // holds -O^T
      tc_fence_before_sync();
      mbar_arrive(&o_empty[ob]);  // the TMEM tile may be overwritten now
      if (v < DIN && p.out) {  // (no output buffer: a forward run for its states only)
        OutT* out = static_cast<OutT*>(p.out) + (size_t)(tok0 + CH * (jb + j)) * H * DIN +
                    (size_t)h * DIN + v;
#pragma unroll
        for (int r = 0; r < CH; ++r)
          if (r < valid && (!SCAN || outputs)) store_out(out + (size_t)r * H * DIN, -p.scale * o[r]);
      }
    }
  } else {
    // ---------------- chain warps: decay, U^T and S^T operands, final state
    // initial state: thread (v, half) holds S^T[v][64 half .. 64 half + 63]
    const int c_lo = 64 * half;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
      float s0[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int c = c_lo + c0 + jj;
        s0[jj] = ident ? (c == v && c < DIN ? 1.f : 0.f)
                       : (s_in && c < DIN && v < DIN) ? s_in[(size_t)c * DIN + v] : 0.f;
      }
      tmem_st16(tl + TB_S + c_lo + c0, s0);
      st8h(layout_addr(ST, v, c_lo + c0), s0);
      st8h(layout_addr(ST, v, c_lo + c0 + 8), s0 + 8);
    }
    tmem_st_wait();
    bool ok = true;
    // A checkpoint due before chunk j is stored from the fp32 state that
    // chunk's decay loads, while the tensor core runs: off the chain.
    float* ck = nullptr;
    for (int j = 0; j < nchunks; ++j) {
      // invariant: ST = fp16(S_j) written by this thread; TMEM S = S_j
      const int buf = j & 1, ob = j & 1;
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(st_ready);
      if (!(ok = mbar_wait(&full[buf], (j >> 1) & 1))) break;
      {  // decay the fp32 state by this chunk's e^{g_C} while the tensor core runs
        const float* gam = gamma_of(buf);
        float sv[64];
        tmem_ld64(tl + TB_S + 64 * half, sv);
        if (ck) {  // S[c][v] = S^T[v][c]
#pragma unroll
          for (int c0 = 0; c0 < 64; ++c0)
            if (c_lo + c0 < DIN) ck[(size_t)(c_lo + c0) * DIN + v] = sv[c0];
          ck = nullptr;
        }
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          float sd[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) sd[jj] = sv[c0 + jj] * gam[64 * half + c0 + jj];
          tmem_st16(tl + TB_S + 64 * half + c0, sd);
        }
        tmem_st_wait();
      }
      if (!(ok = mbar_wait(mma_a, j & 1))) break;
      tc_fence_after_sync();
      {  // U^T = U~^T - S^T W^T (fp16 operand): this thread's 32 tokens
        float u[32], w[32];
        const uint32_t tu = tl + TB_UT + 64 * buf + 32 * half, tw = tl + TB_D + 128 * ob + 32 * half;
        tmem_ld16(tu, *reinterpret_cast<float(*)[16]>(u));
        tmem_ld16(tu + 16, *reinterpret_cast<float(*)[16]>(u + 16));
        tmem_ld16(tw, *reinterpret_cast<float(*)[16]>(w));
        tmem_ld16(tw + 16, *reinterpret_cast<float(*)[16]>(w + 16));
        tmem_ld_wait();
        if (SCAN && kind == 1) {  // no values: U = -S W^T alone
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = w[i];
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] += w[i];
        }
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += 8) st8h(layout_addr(UT, v, 32 * half + r0), u + r0);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(ut_ready);
      if (!(ok = mbar_wait(mma_b, j & 1))) break;
      tc_fence_after_sync();
      {  // the fp16 state operand for the next chunk (and the final state)
        float sv[64];
        tmem_ld64(tl + TB_S + 64 * half, sv);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 8) st8h(layout_addr(ST, v, c_lo + c0), sv + c0);
        if (j + 1 == nchunks && s_out && v < DIN) {  // S[c][v] = S^T[v][c]
#pragma unroll
          for (int c0 = 0; c0 < 64; ++c0)
            if (c_lo + c0 < DIN) s_out[(size_t)(c_lo + c0) * DIN + v] = sv[c0];
        }
        const int done = jb + j + 1;  // chunks of the sequence finished
        if (p.ckpt && done % p.ckpt_every == 0 && done / p.ckpt_every <= p.n_ckpt && v < DIN) {
          float* cp = p.ckpt + ((size_t)(n * p.n_ckpt + done / p.ckpt_every - 1) * H + h) * DIN * DIN;
          if (j + 1 < nchunks) {
            ck = cp;  // with the next chunk's decay
          } else {
#pragma unroll
            for (int c0 = 0; c0 < 64; ++c0)
              if (c_lo + c0 < DIN) cp[(size_t)(c_lo + c0) * DIN + v] = sv[c0];
          }
        }
      }
    }
    if (!ok) {
      fail();
    } else {
      // An fp16 operand that overflowed (a state entry or a correction u
      // beyond the fp16 range) turns into inf / NaN in every later state, so
      // one check of the range's last state, after the chain, catches it.
      float sv[64];
      tmem_ld64(tl + TB_S + 64 * half, sv);
      bool in_range = true;
#pragma unroll
      for (int c0 = 0; c0 < 64; ++c0) in_range &= fabsf(sv[c0]) <= kOperandMax;
      if (!in_range) *s_range = 1;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (tid == 0 && *s_range) set_status(8);
  if (warp == 0) tmem_dealloc(tmem, TB_COLS);
}

// The state pass of chain (sequence n, head h) in the fused launch, run by
// the first B_THREADS threads of its CTA (barrier: named barrier 1): the
// algorithm of kda_state_kernel above, with the records taken from the ring
// once stage 1 has published them.  (The plain kernel keeps its own copy of
// the code: compiled as one kernel function reading its own parameters, its
// chain loop measured faster than in any shared form.)
template <int DIN, typename OutT>
__device__ __forceinline__ void fused_state_body(const CUtensorMap& tm_v, const StateParams& p,
                                                 const FusedRing& ring, uint8_t* smem_raw,
                                                 const int tid, const int n, const int h) {
  constexpr bool SCAN = false, RING = false, FUSED = true;
  const int warp = tid >> 5;
  const int half = (warp >> 2) & 1;           // chain warps: which half of the columns
  const int v = 32 * (warp & 3) + (tid & 31);  // TMEM lane = value channel
  const int H = p.H;
  auto csync = [&]() {
    if (FUSED)
      named_sync(1, B_THREADS);
    else
      __syncthreads();
  };
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sbp = smem_raw + (sb - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sbp + B_MISC);  // [2] record + v tile landed
  uint64_t* mma_a = full + 2;     // D = -S^T [W; q e^g]^T done
  uint64_t* mma_b = full + 3;     // S update and the rest of O done
  uint64_t* o_full = full + 4;    // [2] output tile ready
  uint64_t* o_empty = full + 6;   // [2] output tile drained
  uint64_t* st_ready = full + 8;  // chain -> issuer: S^T operand written
  uint64_t* ut_ready = full + 9;  // chain -> issuer: U^T operand written, state decayed
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sbp + B_MISC + 96);
  int* s_abort = reinterpret_cast<int*>(sbp + B_MISC + 100);
  int* s_range = reinterpret_cast<int*>(sbp + B_MISC + 104);

  int tok0, len, base;
  if (p.plan) {
    tok0 = p.plan[p.n_seq + 1 + n];
    len = p.plan[2 * p.n_seq + 1 + n];
    base = p.plan[n];
  } else {
    tok0 = n * p.T;
    len = p.T;
    base = FUSED  ? n * ring.R
           : RING ? n * p.rec_stride + p.rec_shift
                  : n * ((p.T + CH - 1) / CH);
  }
  const int nch_seq = len > 0 ? (len + CH - 1) / CH : 0;
  const int jb = p.j_lo, nchunks = max(0, min(p.j_hi, nch_seq) - jb);  // j below is jb + local
  const size_t sbase = (size_t)(n * H + h) * DIN * DIN;
  // the walk this CTA does: kind 0 the plain recurrence with outputs, 1 the
  // transition (identity start, no values, no outputs), 2 the zero-start
  // state (no outputs); and where its first state comes from and its last
  // state goes
  const int seg = SCAN ? n % p.segs : 0;
  const size_t real = (size_t)((SCAN ? n / p.segs : n) * H + h) * DIN * DIN;
  float* carry = p.carry ? p.carry + 0 + sbase : nullptr;
  int kind = 0;
  if (SCAN && p.phase == 1 && seg > 0) kind = 2;
  if (SCAN && (false || (p.phase == 2 && seg == 0))) return;
  const bool last_range = jb + nchunks == nch_seq;
  const float* s_in;
  float* s_out;
  if (!SCAN) {
    s_in = jb == 0 ? (p.s0 ? p.s0 + sbase : nullptr) : carry;
    s_out = last_range ? (p.s1 ? p.s1 + sbase : nullptr) : carry;
  } else if (p.phase == 1) {
    s_in = jb > 0 ? carry : (kind == 0 && p.s0 ? p.s0 + real : nullptr);
    s_out = carry;
  } else {
    s_in = carry;
    s_out = last_range && seg == p.segs - 1 && p.s1 ? p.s1 + real : nullptr;
  }
  const bool ident = SCAN && kind == 1 && jb == 0;  // the transition walk starts from I
  const bool outputs = !SCAN || kind == 0;
  if (nchunks == 0) {  // nothing in this range; a sequence with no tokens keeps its state
    if (jb == 0 && nch_seq == 0 && s_out)
      for (int i = tid; i < DIN * DIN; i += B_THREADS)
        s_out[i] = ident ? (i / DIN == i % DIN ? 1.f : 0.f) : (s_in ? s_in[i] : 0.f);
    return;
  }
  constexpr uint32_t kVBytes = (DIN / 64) * 8192u;
  const int chain = n * H + h;
  // The loads of chunk jb + j into buffer buf.  Fused: once stage 1 has
  // published that record (false if it never does).
  // seen: the record's ready flag as read earlier (fused)
  auto ready_flag = [&](int j) { return ring.ready + chain * ring.ready_stride + (jb + j) % ring.R; };
  auto issue_loads = [&](int j, int buf, int seen) -> bool {
    const int jr = FUSED ? (jb + j) % ring.R : jb + j;
    if (FUSED) {
      if (!poll_at_least(ready_flag(j), jb + j + 1, seen)) return false;
      fence_proxy_async_global();
    }
    const uint8_t* rec = p.records + ((size_t)(base + jr) * H + h) * REC_BYTES;
    uint8_t* dst = sbp + (buf ? B_REC1 : B_REC0);
    uint8_t* vdst = sbp + (buf ? B_V1 : B_V0);
    mbar_arrive_expect_tx(&full[buf], REC_LOAD + (SCAN && kind == 1 ? 0u : kVBytes));
    bulk_g2s(dst, rec, REC_LOAD, &full[buf]);
    if (!SCAN || kind != 1) {
#pragma unroll
      for (int b = 0; b < DIN / 64; ++b)
        tma_load_3d(vdst + b * 8192, &tm_v, &full[buf], b * 64, h, tok0 + CH * (jb + j));
    }
    return true;
  };
  // fused: the records of chunks below jb + upto are in shared memory (their
  // copies have completed), so their slots are free for stage 1.  A relaxed
  // store: nothing the chain still reads depends on it, and a release would
  // wait for this thread's copies in flight.
  auto release = [&](int upto) {
    if (FUSED) st_relaxed_gpu(ring.consumed + chain * kFlagLine, jb + upto);
  };
  auto gamma_of = [&](int buf) {
    return reinterpret_cast<const float*>(sbp + (buf ? B_REC1 : B_REC0) + REC_G);
  };

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(mma_a, 1);
    mbar_init(mma_b, 1);
    mbar_init(&o_full[0], 1);
    mbar_init(&o_full[1], 1);
    mbar_init(&o_empty[0], B_OUTPUT);
    mbar_init(&o_empty[1], B_OUTPUT);
    mbar_init(st_ready, B_CHAIN);
    mbar_init(ut_ready, B_CHAIN);
    mbar_fence_init();
    *s_abort = 0;
    *s_range = 0;
    if (!FUSED) {  // (fused: the issuer makes them, once stage 1 has published)
      if (nchunks > 0) issue_loads(0, 0, 0);
      if (nchunks > 1) issue_loads(1, 1, 0);
    }
  }
  if (DIN == 64) {
    for (uint32_t off = tid * 16; off < 8192; off += B_THREADS * 16) {
      st_shared_v4(sb + B_V0 + 8192 + off, 0, 0, 0, 0);
      st_shared_v4(sb + B_V1 + 8192 + off, 0, 0, 0, 0);
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_s, TB_COLS);
    if (!FUSED) tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  csync();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_base_s;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const OperandLayout ST = kmajor(sb + B_ST, 16384);  // M = v, K = c
  const OperandLayout UT = kmajor(sb + B_UT, 0);      // M = v, K = i
  auto fail = [&]() {
    *s_abort = 1;
    set_status(6);
  };

  if (warp == B_THREADS / 32 - 1) {
    // ---------------- issuer: one lane issues every MMA and every load
    if ((tid & 31) == 0 && nchunks > 0) {
      constexpr uint32_t ID_V = make_idesc(128, 64, true, false);                 // bf16
      constexpr uint32_t ID_O2 = make_idesc(128, 64, false, true, true, true);    // fp16, -A
      constexpr uint32_t ID_S = make_idesc(128, 128, false, false, false, true);  // fp16
      // M3 of chunk j, U~^T = V^T (T diag beta)^T, needs no state: it is
      // issued as soon as record j lands, ahead of the chain's own products.
      auto issue_m3 = [&](int j) {
        if (SCAN && kind == 1) return;  // no values: U~ = 0
        const int b = j & 1;
        const uint32_t rb = sb + (b ? B_REC1 : B_REC0), vb = sb + (b ? B_V1 : B_V0);
        const uint64_t dva = layout_desc(mnmajor(vb, 8192), 0, 0);
        const uint64_t dtb = layout_desc(kmajor(rb + REC_TB, 0), 0, 0);
#pragma unroll
        for (int k0 = 0; k0 < CH; k0 += 16)
          umma_bf16(tmem + TB_UT + 64 * b, desc_adv(dva, k0, true), desc_adv(dtb, k0, false),
                    ID_V, k0 > 0);
      };
      int issued = FUSED ? 0 : min(nchunks, 2), landed = 0;  // record loads issued / seen complete
      int seen_next = 0;  // fused: the ready flag of the next load, read ahead
      bool ok = true;
      if (FUSED) {
        ok = issue_loads(0, 0, ld_relaxed_gpu(ready_flag(0)));
        issued = ok ? 1 : 0;
        if (ok && nchunks > 1) {
          ok = issue_loads(1, 1, ld_relaxed_gpu(ready_flag(1)));
          issued += ok ? 1 : 0;
        }
      }
      ok = ok && mbar_wait(&full[0], 0);
      if (ok) {
        landed = 1;
        release(1);
        tc_fence_after_sync();
        issue_m3(0);
      }
      for (int j = 0; j < nchunks && ok; ++j) {
        const int buf = j & 1, ob = j & 1;
        const uint32_t rb = sb + (buf ? B_REC1 : B_REC0);
        const uint32_t td = tmem + TB_D + 128 * ob;
        if (!(ok = mbar_wait(st_ready, j & 1))) break;
        if (j >= 2 && !(ok = mbar_wait(&o_empty[ob], ((j - 2) >> 1) & 1))) break;
        tc_fence_after_sync();
        {  // M4, D = -S^T W^T, alone (N = 64): the chain waits only for it.  The
           // first half of M5, -S^T (q e^g)^T, follows into the next 64 columns
           // and runs while the chain forms U^T.
          const uint64_t dst = layout_desc(ST, 0, 0);
          const uint64_t dw = layout_desc(mnmajor(rb + REC_WT, 16384), 0, 0);
          const uint64_t dq = layout_desc(mnmajor(rb + REC_QT, 16384), 0, 0);
#pragma unroll
          for (int k0 = 0; k0 < DP; k0 += 16)
            umma_bf16(td, desc_adv(dst, k0, false, 16384), desc_adv(dw, k0, true), ID_O2, k0 > 0);
          umma_commit(mma_a);
          // fused: read the ready flag of chunk j + 2 now; it is needed only
          // once chunk j's products are done, and the load runs meanwhile
          if (FUSED && j + 2 < nchunks) seen_next = ld_relaxed_gpu(ready_flag(j + 2));
#pragma unroll
          for (int k0 = 0; k0 < DP; k0 += 16)
            umma_bf16(td + 64, desc_adv(dst, k0, false, 16384), desc_adv(dq, k0, true), ID_O2,
                      k0 > 0);
        }
        if (!(ok = mbar_wait(ut_ready, j & 1))) break;
        tc_fence_after_sync();
        {
          const uint64_t dut = layout_desc(UT, 0, 0);
          const uint64_t daq = layout_desc(mnmajor(rb + REC_AQ, 8192), 0, 0);
          const uint64_t dkb = layout_desc(kmajor(rb + REC_KBAR, 0), 0, 0);
          // M6 first: the chain waits only for the state update; the second
          // half of M5 (the output) runs while the chain rebuilds S^T
#pragma unroll
          for (int k0 = 0; k0 < CH; k0 += 16)
            umma_bf16(tmem + TB_S, desc_adv(dut, k0, false), desc_adv(dkb, k0, false), ID_S, 1);
          umma_commit(mma_b);
#pragma unroll
          for (int k0 = 0; k0 < CH; k0 += 16)
            umma_bf16(td + 64, desc_adv(dut, k0, false), desc_adv(daq, k0, true), ID_O2, 1);
          umma_commit(&o_full[ob]);
        }
        if (j + 2 < nchunks) {  // buffer buf is consumed once every product of chunk j is done
          if (!(ok = mbar_wait(&o_full[ob], (j >> 1) & 1))) break;
          fence_proxy_async_smem();
          if (!(ok = issue_loads(j + 2, buf, seen_next))) break;
          ++issued;
        }
        if (j + 1 < nchunks) {
          if (!(ok = mbar_wait(&full[buf ^ 1], ((j + 1) >> 1) & 1))) break;
          ++landed;
          release(j + 2);
          tc_fence_after_sync();
          issue_m3(j + 1);
        }
      }
      if (!ok) {
        fail();
        // let copies already issued land before the CTA's memory goes away
        for (int r = landed; r < issued; ++r) mbar_wait(&full[r & 1], (r >> 1) & 1, 100000000ull);
      }
    }
  } else if (warp >= B_CHAIN / 32) {
    // ---------------- output warps: thread = value channel v, all 64 tokens
    for (int j = 0; j < nchunks; ++j) {
      const int ob = j & 1;
      if (!mbar_wait(&o_full[ob], (j >> 1) & 1)) {
        fail();
        break;
      }
      tc_fence_after_sync();
      const int valid = min(CH, len - CH * (jb + j));
      float o[64];
      tmem_ld64(tl + TB_D + 128 * ob + 64, o);  // holds -O^T
      tc_fence_before_sync();
      mbar_arrive(&o_empty[ob]);  // the TMEM tile may be overwritten now
      if (v < DIN && p.out) {  // (no output buffer: a forward run for its states only)
        OutT* out = static_cast<OutT*>(p.out) + (size_t)(tok0 + CH * (jb + j)) * H * DIN +
                    (size_t)h * DIN + v;
#pragma unroll
        for (int r = 0; r < CH; ++r)
          if (r < valid && (!SCAN || outputs)) store_out(out + (size_t)r * H * DIN, -p.scale * o[r]);
      }
    }
  } else {
    // ---------------- chain warps: decay, U^T and S^T operands, final state
    // initial state: thread (v, half) holds S^T[v][64 half .. 64 half + 63]
    const int c_lo = 64 * half;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
      float s0[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int c = c_lo + c0 + jj;
        s0[jj] = ident ? (c == v && c < DIN ? 1.f : 0.f)
                       : (s_in && c < DIN && v < DIN) ? s_in[(size_t)c * DIN + v] : 0.f;
      }
      tmem_st16(tl + TB_S + c_lo + c0, s0);
      st8h(layout_addr(ST, v, c_lo + c0), s0);
      st8h(layout_addr(ST, v, c_lo + c0 + 8), s0 + 8);
    }
    tmem_st_wait();
    bool ok = true;
    // A checkpoint due before chunk j is stored from the fp32 state that
    // chunk's decay loads, while the tensor core runs: off the chain.
    float* ck = nullptr;
    for (int j = 0; j < nchunks; ++j) {
      // invariant: ST = fp16(S_j) written by this thread; TMEM S = S_j
      const int buf = j & 1, ob = j & 1;
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(st_ready);
      if (!(ok = mbar_wait(&full[buf], (j >> 1) & 1))) break;
      {  // decay the fp32 state by this chunk's e^{g_C} while the tensor core runs
        const float* gam = gamma_of(buf);
        float sv[64];
        tmem_ld64(tl + TB_S + 64 * half, sv);
        if (ck) {  // S[c][v] = S^T[v][c]
#pragma unroll
          for (int c0 = 0; c0 < 64; ++c0)
            if (c_lo + c0 < DIN) ck[(size_t)(c_lo + c0) * DIN + v] = sv[c0];
          ck = nullptr;
        }
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          float sd[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) sd[jj] = sv[c0 + jj] * gam[64 * half + c0 + jj];
          tmem_st16(tl + TB_S + 64 * half + c0, sd);
        }
        tmem_st_wait();
      }
      if (!(ok = mbar_wait(mma_a, j & 1))) break;
      tc_fence_after_sync();
      {  // U^T = U~^T - S^T W^T (fp16 operand): this thread's 32 tokens
        float u[32], w[32];
        const uint32_t tu = tl + TB_UT + 64 * buf + 32 * half, tw = tl + TB_D + 128 * ob + 32 * half;
        tmem_ld16(tu, *reinterpret_cast<float(*)[16]>(u));
        tmem_ld16(tu + 16, *reinterpret_cast<float(*)[16]>(u + 16));
        tmem_ld16(tw, *reinterpret_cast<float(*)[16]>(w));
        tmem_ld16(tw + 16, *reinterpret_cast<float(*)[16]>(w + 16));
        tmem_ld_wait();
        if (SCAN && kind == 1) {  // no values: U = -S W^T alone
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = w[i];
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] += w[i];
        }
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += 8) st8h(layout_addr(UT, v, 32 * half + r0), u + r0);
        if (ring.u_out && v < DIN) {  // this thread's value channel of 32 tokens
          const int t0 = CH * (jb + j) + 32 * half;
          float* uo = ring.u_out + ((size_t)(tok0 + t0) * H + h) * DIN + v;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (t0 + i < len) uo[(size_t)i * H * DIN] = u[i];
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(ut_ready);
      if (!(ok = mbar_wait(mma_b, j & 1))) break;
      tc_fence_after_sync();
      {  // the fp16 state operand for the next chunk (and the final state)
        float sv[64];
        tmem_ld64(tl + TB_S + 64 * half, sv);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 8) st8h(layout_addr(ST, v, c_lo + c0), sv + c0);
        if (j + 1 == nchunks && s_out && v < DIN) {  // S[c][v] = S^T[v][c]
#pragma unroll
          for (int c0 = 0; c0 < 64; ++c0)
            if (c_lo + c0 < DIN) s_out[(size_t)(c_lo + c0) * DIN + v] = sv[c0];
        }
        const int done = jb + j + 1;  // chunks of the sequence finished
        if (p.ckpt && done % p.ckpt_every == 0 && done / p.ckpt_every <= p.n_ckpt && v < DIN) {
          float* cp = p.ckpt + ((size_t)(n * p.n_ckpt + done / p.ckpt_every - 1) * H + h) * DIN * DIN;
          if (j + 1 < nchunks) {
            ck = cp;  // with the next chunk's decay
          } else {
#pragma unroll
            for (int c0 = 0; c0 < 64; ++c0)
              if (c_lo + c0 < DIN) cp[(size_t)(c_lo + c0) * DIN + v] = sv[c0];
          }
        }
      }
    }
    if (!ok) {
      fail();
    } else {
      // An fp16 operand that overflowed (a state entry or a correction u
      // beyond the fp16 range) turns into inf / NaN in every later state, so
      // one check of the range's last state, after the chain, catches it.
      float sv[64];
      tmem_ld64(tl + TB_S + 64 * half, sv);
      bool in_range = true;
#pragma unroll
      for (int c0 = 0; c0 < 64; ++c0) in_range &= fabsf(sv[c0]) <= kOperandMax;
      if (!in_range) *s_range = 1;
    }
  }
  tc_fence_before_sync();
  csync();
  if (tid == 0 && *s_range) set_status(8);
  if (warp == 0) tmem_dealloc(tmem, TB_COLS);
}

// The whole prefill of fixed-length sequences in one cooperative launch of
// one CTA per SM (see FusedRing): CTA c < B H walks chain c with its first
// B_THREADS threads, every other CTA runs two stage-1 bodies, one per
// 256-thread half, on its two halves of shared memory and tensor memory.
template <int DIN, typename OutT>
__global__ void __launch_bounds__(F_THREADS, 1)
    kda_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ IntraParams ip, const __grid_constant__ StateParams sp,
                     const __grid_constant__ FusedRing ring) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((int)blockIdx.x < sp.n_seq * sp.H) {
    if (threadIdx.x < B_THREADS)
      fused_state_body<DIN, OutT>(tm_v, sp, ring, smem_raw, threadIdx.x, (int)blockIdx.x / sp.H,
                                  (int)blockIdx.x % sp.H);
    return;
  }
  const int part = threadIdx.x / A_THREADS;
  intra_body<DIN, false, false, true, const IntraParams&>(tm_q, tm_k, tm_g, ip, ring,
                                                          smem_raw + part * A_SMEM,
                                                          threadIdx.x % A_THREADS, 1 + part);
}

// Packed sequences: the plan every later kernel reads instead of cu_seqlens,
//   plan[n]             = sum_{m < n} ceil(len_m / 64)   (n = 0..N, record offsets)
//   plan[N + 1 + n]     = start_n,   plan[2N + 1 + n] = len_n   (n < N)
// with each sequence clamped into [0, T_total) and to at most max_len tokens
// (the work list is sized by max_len), so that no kernel addresses a token
// or a record outside the caller's buffers whatever cu_seqlens holds.  A
// sequence that had to be clamped -- cu[0] != 0, a decreasing offset, an
// offset past T_total, or a length above max_len -- is reported as an
// invalid argument in the status word.
__global__ void __launch_bounds__(1024) kda_plan_kernel(const int* __restrict__ cu, int N,
                                                        int max_len, int T_total,
                                                        int* __restrict__ plan) {
  __shared__ int warp_tot[32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int start = 0; start <= N; start += 1024) {
    const int i = start + tid;
    int cnt = 0;
    if (i < N) {
      const int a = cu[i], b = cu[i + 1];
      const int s0 = min(max(a, 0), T_total);
      const int e0 = min(max(b, s0), T_total);
      const int len = min(e0 - s0, max_len);
      if ((i == 0 && a != 0) || b < a || b > T_total || b - a > max_len) set_status(1);
      plan[N + 1 + i] = s0;
      plan[2 * N + 1 + i] = len;
      cnt = len > 0 ? (len + CH - 1) / CH : 0;
    }
    int x = cnt;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
      int t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int excl = carry_s + (w > 0 ? warp_tot[w - 1] : 0) + x - cnt;
    if (i <= N) plan[i] = excl;
    __syncthreads();
    if (tid == 0) carry_s += warp_tot[31];
    __syncthreads();
  }
}

// Segment scan over fixed-length sequences: segment q of sequence b is
// sequence b * segs + q of the work list, seg_tok tokens (whole chunks) from
// token q * seg_tok of sequence b, the last one shorter.  Its records are
// those of the same chunks of the unsegmented problem.
__global__ void __launch_bounds__(256) kda_segment_plan_kernel(int B, int T, int seg_tok, int segs,
                                                               int* __restrict__ plan) {
  const int N = B * segs, nc = (T + CH - 1) / CH, lc = seg_tok / CH;
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n <= N; n += blockDim.x * gridDim.x) {
    if (n == N) {
      plan[N] = B * nc;
      continue;
    }
    const int b = n / segs, q = n % segs;
    plan[n] = b * nc + q * lc;
    plan[N + 1 + n] = b * T + q * seg_tok;
    plan[2 * N + 1 + n] = min(seg_tok, T - q * seg_tok);
  }
}

// The scan of a sequence cut into segments (the orkas.ai page, "Kimi K3
// architecture", section "Die Rechnung landet in der
// Bereitstellungsinfrastruktur": each segment reduces to a cumulative
// transition and a zero-start state, composed by a prefix scan).  With M_q,
// Z_q segment q's transition and zero-start state (planes 1 and 0 of the
// carried states) and E_1 the state after segment 0 (plane 0 of segment 0),
//   E_{q+1} = M_q E_q + Z_q,   q = 1 .. segs - 2,
// in fp32.  E_q replaces Z_q in plane 0, where the second walk of segment q
// starts from it.  One CTA per (sequence, head).
template <int DIN>
constexpr uint32_t kScanSmem = (uint32_t)DIN * (DIN + 4) * 4u + (uint32_t)DIN * (32 + 4) * 4u;

// One CTA per (sequence, head, block of 32 state columns): E's columns are
// independent under the left multiplication by M.
template <int DIN>
__global__ void __launch_bounds__(256) kda_scan_combine_kernel(float* __restrict__ carry, int n_seq,
                                                               int segs, int H) {
  extern __shared__ float scan_sm[];
  constexpr int LD = DIN + 4, LC = 32 + 4;  // row strides in floats
  constexpr int TR = DIN / 32;              // each thread: TR rows x 4 columns of the product
  float* Ms = scan_sm;                      // M_q, DIN x DIN
  float* Cs = scan_sm + DIN * LD;           // E_q, DIN x 32 (this CTA's columns)
  const int h = blockIdx.x, b = blockIdx.y, col0 = 32 * blockIdx.z, tid = threadIdx.x;
  const size_t mat = (size_t)DIN * DIN, plane = (size_t)n_seq * H * mat;
  auto at = [&](int z, int q) { return carry + z * plane + ((size_t)(b * segs + q) * H + h) * mat; };
  const int r0 = (tid / 8) * TR, c0 = (tid % 8) * 4;
  for (int i = tid; i < DIN * 32; i += 256) Cs[(i / 32) * LC + i % 32] = at(0, 0)[(i / 32) * DIN + col0 + i % 32];
  __syncthreads();
  for (int q = 1; q < segs; ++q) {
    float* Zg = at(0, q);
    float acc[TR][4];
    const bool more = q + 1 < segs;  // E_{q+1} is needed
    if (more) {
      const float* Mg = at(1, q);
      for (int i = tid; i < DIN * DIN; i += 256) Ms[(i / DIN) * LD + i % DIN] = Mg[i];
      __syncthreads();
#pragma unroll
      for (int i = 0; i < TR; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = Zg[(size_t)(r0 + i) * DIN + col0 + c0 + j];
      for (int k = 0; k < DIN; ++k) {
        const float4 x = *reinterpret_cast<const float4*>(Cs + k * LC + c0);
#pragma unroll
        for (int i = 0; i < TR; ++i) {
          const float a = Ms[(r0 + i) * LD + k];
          acc[i][0] = fmaf(a, x.x, acc[i][0]);
          acc[i][1] = fmaf(a, x.y, acc[i][1]);
          acc[i][2] = fmaf(a, x.z, acc[i][2]);
          acc[i][3] = fmaf(a, x.w, acc[i][3]);
        }
      }
    }
    __syncthreads();  // every read of Z_q's columns and of E_q in shared memory is done
    for (int i = tid; i < DIN * 32; i += 256)
      Zg[(size_t)(i / 32) * DIN + col0 + i % 32] = Cs[(i / 32) * LC + i % 32];  // E_q
    __syncthreads();
    if (more) {
#pragma unroll
      for (int i = 0; i < TR; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) Cs[(r0 + i) * LC + c0 + j] = acc[i][j];
    }
    __syncthreads();
  }
}

template <typename K>
cudaError_t set_smem(K kern, uint32_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// SM count of the current device, cached per device.
int g_sms[64];
std::mutex g_sms_mu;
cudaError_t device_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_sms_mu);
  if (!g_sms[dev]) {
    e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  *sms = g_sms[dev];
  return cudaSuccess;
}

// Chunks per segment of the overlapped schedule: about eight segments, a
// multiple of 16 chunks, at least 32.
int segment_chunks(int nc_max) {
  const int s = (nc_max + 7) / 8;
  return s < 32 ? 32 : (s + 15) / 16 * 16;
}

// Fixed lengths in the overlapped schedule (no scan) keep the records in a
// ring of two segments: stage 1 of segment k + 2 starts only after the state
// pass of segment k has finished (it is a programmatic dependent of the
// state pass of segment k + 1, which starts after stage 1 of segment k + 1,
// whose grid completes after the state pass of segment k).  The segment is
// at most kRingMaxSegment chunks, and less where the ring would exceed
// kRingBudget, so the workspace stops growing with T.
constexpr int kRingMaxSegment = 128;
constexpr size_t kRingBudget = (size_t)1 << 30;
// The ring is taken only where one record per chunk would pass this size.
constexpr size_t kRingThreshold = (size_t)4 << 30;
bool ring_records(int n_seq, int nc, int H) {
  return (size_t)n_seq * (size_t)nc * (size_t)H * REC_BYTES > kRingThreshold;
}
int ring_segment_chunks(int nc_max, int chains) {
  const long long cap = (long long)(kRingBudget / (2ull * (unsigned)chains * REC_BYTES)) / 16 * 16;
  const long long seg = std::min<long long>(std::min(segment_chunks(nc_max), kRingMaxSegment), cap);
  return (int)std::max<long long>(32, seg);
}

// Records per chain in the fused launch's ring (at most the chunks of a
// sequence): 16 chunks x 32 heads x 65 KB is 33 MB, well inside L2.
constexpr int kFusedRing = 16;
// KDA_SCHEDULE, read on every call, overrides the choice below for
// comparisons: "rounds" keeps fixed-length calls on the two-kernel round
// schedule, "fused" takes the fused launch wherever it can run (chains on at
// most half the SMs).  Returns 'r', 'f' or 0.
char schedule_forced() {
  const char* e = std::getenv("KDA_SCHEDULE");
  if (!e) return 0;
  if (std::strcmp(e, "rounds") == 0) return 'r';
  if (std::strcmp(e, "fused") == 0) return 'f';
  return 0;
}
// Where the fused launch is the faster schedule (measured on the fixed-length
// prefill, d = 128, against the round schedule): its chains run about as
// fast as the plain state pass, but its stage 1, on the SMs the chains leave
// and with each record's publication to pay for, keeps up with them only
// while they are few.  With up to sms / 9 chains (16 of 152 SMs) it wins at
// every length tried (up to 64k tokens, 4-10 % from 8k on); with up to sms /
// 4 (32 heads) it wins up to 512 chunks (8-25 %) and loses 1 % at 1024; with
// 64 chains it loses 25-50 %.
bool use_fused(bool eligible, int chains, int nc, int sms) {
  const char f = schedule_forced();
  if (!eligible || f == 'r') return false;
  if (f == 'f') return 2 * chains <= sms;
  return 9 * chains <= sms || (4 * chains <= sms && nc <= 512);
}

// The overlapped schedule pays off for sequences of at least 128 chunks
// (8192 tokens) and few long-lived state chains: stage 2 must leave stage 1
// at least half the SMs.
bool use_overlap(int n_states, int nc_max, int sms) {
  return n_states <= sms / 2 && nc_max >= 128;
}

template <int DIN, typename OutT>
cudaError_t launch_stages(const ChunkProblem& pr, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tg, int* plan,
                          uint8_t* records, float* carry, int* grid_done, int nc_max,
                          bool allow_overlap, cudaStream_t stream) {
  // the shared-memory opt-in is a per-device function attribute; setting it
  // on every call costs next to nothing
  cudaError_t e = set_smem(kda_intra_kernel<DIN, false>, A_SMEM);
  if (e == cudaSuccess) e = set_smem(kda_intra_kernel<DIN, true>, A_SMEM);
  if (e == cudaSuccess) e = set_smem(kda_state_kernel<DIN, OutT, false>, B_SMEM);
  if (e == cudaSuccess && pr.scan_segs > 1) e = set_smem(kda_state_kernel<DIN, OutT, true>, B_SMEM);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = device_sms(&sms);
  if (e != cudaSuccess) return e;

  // Two CTAs per SM.  dependent: a programmatic dependent launch of the state
  // pass just enqueued (it may start once that grid's CTAs are all resident).
  // persistent: two CTAs per SM take items from a counter, so CTAs that start
  // late (on SMs a state pass holds) take fewer; else one CTA per item.
  int ring = 0;  // records per sequence in a ring (set with the schedule below), 0 = all
  auto intra = [&](int j_lo, int seg_len, bool dependent, bool persistent) -> cudaError_t {
    const long long items = (long long)pr.n_seq * seg_len * pr.H;
    IntraParams ip{static_cast<const __nv_bfloat16*>(pr.beta), records, plan,
                   pr.T, pr.n_seq, pr.H, pr.check_decay ? 1 : 0, j_lo, seg_len, (int)items,
                   ring ? ring : (pr.T + CH - 1) / CH, ring ? j_lo % ring - j_lo : 0,
                   persistent ? grid_done : nullptr};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(persistent ? std::min<long long>(items, 2LL * sms) : items));
    cfg.blockDim = dim3(A_THREADS);
    cfg.dynamicSmemBytes = A_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    if (ring) return cudaLaunchKernelEx(&cfg, kda_intra_kernel<DIN, false, true>, tq, tk, tg, ip);
    return pr.diag_per_pair ? cudaLaunchKernelEx(&cfg, kda_intra_kernel<DIN, true>, tq, tk, tg, ip)
                            : cudaLaunchKernelEx(&cfg, kda_intra_kernel<DIN, false>, tq, tk, tg, ip);
  };
  const int segs = pr.scan_segs > 1 ? pr.scan_segs : 1;
  auto state = [&](int j_lo, int j_hi, int phase) -> cudaError_t {
    StateParams sp{records, pr.initial_state, pr.final_state, carry, pr.out, plan,
                   pr.T, pr.n_seq, pr.H, j_lo, j_hi, pr.scale,
                   pr.ckpt, pr.ckpt_every_chunks, pr.n_ckpt, segs, phase,
                   // in a ring, chunk j of this range sits at n ring + j % ring: the
                   // range is one segment starting at a multiple of its length and the
                   // ring holds two, so n ring + (j_lo % ring - j_lo) + j stays inside it
                   ring ? ring : (pr.T + CH - 1) / CH, ring ? j_lo % ring - j_lo : 0};
    const dim3 grid((unsigned)pr.H, (unsigned)pr.n_seq, phase == 1 ? 2 : 1);
    if (phase == 0 && ring)
      kda_state_kernel<DIN, OutT, false, true><<<grid, B_THREADS, B_SMEM, stream>>>(tv, sp);
    else if (phase == 0)
      kda_state_kernel<DIN, OutT, false><<<grid, B_THREADS, B_SMEM, stream>>>(tv, sp);
    else
      kda_state_kernel<DIN, OutT, true><<<grid, B_THREADS, B_SMEM, stream>>>(tv, sp);
    return cudaGetLastError();
  };
  // segment scan, after every segment has been walked: the entry states,
  // then the later segments once more with outputs
  auto finish_scan = [&]() -> cudaError_t {
    if (segs == 1) return cudaSuccess;
    cudaError_t e2 = set_smem(kda_scan_combine_kernel<DIN>, kScanSmem<DIN>);
    if (e2 != cudaSuccess) return e2;
    kda_scan_combine_kernel<DIN><<<dim3((unsigned)pr.H, (unsigned)(pr.n_seq / segs), DIN / 32),
                                   256, kScanSmem<DIN>, stream>>>(carry, pr.n_seq, segs, pr.H);
    e2 = cudaGetLastError();
    if (e2 == cudaSuccess) e2 = state(0, nc_max, 2);
    return e2;
  };
  const int first_phase = segs > 1 ? 1 : 0;

  // Overlapped schedule, all on the caller's stream: segments of chunks,
  //   intra(0), state(0), intra(1)*, state(1), intra(2)*, ...
  // where * marks a programmatic dependent launch.  A state pass holds one
  // SM per (sequence, head) and lets the next segment's intra-chunk stage
  // fill the other SMs while it runs; that stage's grid completes only after
  // the state pass (its last CTA waits for it), so every state pass starts
  // after both the records of its segment and the state carried into it.
  // Stage-2 CTAs that stay resident for most of the call: every (sequence,
  // head) for fixed lengths; for packed sequences about H per multiple of the
  // longest length (short sequences' chains end early and give their SMs back).
  // A segment scan walks 2 segs - 1 chains per (sequence, head); its state
  // passes are short, so they may take up to every SM.
  // The fused single launch (kda_fused_kernel): fixed lengths, no scan, no
  // per-round host copies, not the ablation, with the workspace's counters,
  // where it is the faster schedule (use_fused).  Its ring of records stays
  // in L2.
  const bool fused_ok = !pr.cu_seqlens && segs == 1 && !pr.hooks && !pr.diag_per_pair &&
                        allow_overlap && carry && grid_done;
  // u wanted (the backward's forward): only the fused launch writes it
  if (pr.u_out && !(fused_ok && 2 * pr.n_seq * pr.H <= sms)) return cudaErrorNotSupported;
  if (pr.u_out || use_fused(fused_ok, pr.n_seq * pr.H, nc_max, sms)) {
    const int chains = pr.n_seq * pr.H, R = std::min(kFusedRing, nc_max);
    // flags in the carry (not used by this path): the counter's line, a line
    // per chain for consumed, then each chain's ready slots on lines of their own
    const int ready_stride = (R + kFlagLine - 1) / kFlagLine * kFlagLine;
    int* flags = reinterpret_cast<int*>(carry);
    const FusedRing fr{flags + (size_t)(1 + chains) * kFlagLine, flags + kFlagLine, flags, R,
                       ready_stride, pr.u_out};
    const size_t flag_ints = (size_t)(1 + chains) * kFlagLine + (size_t)chains * ready_stride;
    e = cudaMemsetAsync(flags, 0, flag_ints * sizeof(int), stream);
    if (e != cudaSuccess) return e;
    IntraParams ip{};
    ip.beta = static_cast<const __nv_bfloat16*>(pr.beta);
    ip.records = records;
    ip.T = pr.T;
    ip.n_seq = pr.n_seq;
    ip.H = pr.H;
    ip.check_decay = pr.check_decay ? 1 : 0;
    ip.j_lo = 0;
    ip.seg_len = nc_max;
    ip.n_items = nc_max * chains;
    StateParams sp{};
    sp.records = records;
    sp.s0 = pr.initial_state;
    sp.s1 = pr.final_state;
    sp.out = pr.out;
    sp.T = pr.T;
    sp.n_seq = pr.n_seq;
    sp.H = pr.H;
    sp.j_lo = 0;
    sp.j_hi = nc_max;
    sp.scale = pr.scale;
    sp.ckpt = pr.ckpt;
    sp.ckpt_every = pr.ckpt_every_chunks;
    sp.n_ckpt = pr.n_ckpt;
    sp.segs = 1;
    const auto fused = kda_fused_kernel<DIN, OutT>;
    e = set_smem(fused, F_SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(F_THREADS);
    cfg.dynamicSmemBytes = F_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused, tq, tk, tg, tv, ip, sp, fr);
  }
  const int long_chains = segs > 1 ? (pr.n_seq / segs) * (2 * segs - 1) * pr.H
      : pr.cu_seqlens ? pr.H * (int)(((long long)pr.T_total + pr.T - 1) / std::max(pr.T, 1))
      : pr.n_seq * pr.H;
  const bool overlap = allow_overlap && carry && grid_done &&
                       use_overlap(segs > 1 ? long_chains / 2 : long_chains, nc_max, sms);
  RoundHooks* hooks = segs == 1 && !pr.cu_seqlens ? pr.hooks : nullptr;
  if (!overlap) {
    const bool persistent = grid_done != nullptr;
    if (persistent) e = cudaMemsetAsync(grid_done, 0, 2 * sizeof(int), stream);
    if (e == cudaSuccess && hooks) e = hooks->before_round(0, nc_max, stream);
    if (e == cudaSuccess) e = intra(0, nc_max, false, persistent);
    if (e == cudaSuccess) e = state(0, nc_max, first_phase);
    if (e == cudaSuccess && hooks) e = hooks->after_round(0, nc_max, stream);
    if (e == cudaSuccess) e = finish_scan();
    return e;
  }
  const bool use_ring = !pr.cu_seqlens && segs == 1 && ring_records(pr.n_seq, nc_max, pr.H);
  const int seg = use_ring ? ring_segment_chunks(nc_max, long_chains) : segment_chunks(nc_max);
  if (use_ring) {  // (the per-pair ablation is not offered with a ring)
    ring = 2 * seg;
    e = set_smem(kda_state_kernel<DIN, OutT, false, true>, B_SMEM);
    if (e == cudaSuccess) e = set_smem(kda_intra_kernel<DIN, false, true>, A_SMEM);
    if (e != cudaSuccess) return e;
  }
  e = cudaMemsetAsync(grid_done, 0, 2 * sizeof(int), stream);
  for (int j_lo = 0; e == cudaSuccess && j_lo < nc_max; j_lo += seg) {
    const int len = std::min(seg, nc_max - j_lo);
    if (hooks) e = hooks->before_round(j_lo, len, stream);
    if (e == cudaSuccess) e = intra(j_lo, len, j_lo > 0, true);
    if (e == cudaSuccess) e = state(j_lo, j_lo + len, first_phase);
    if (e == cudaSuccess && hooks) e = hooks->after_round(j_lo, len, stream);
  }
  if (e == cudaSuccess) e = finish_scan();
  return e;
}

}  // namespace

// Counts the long-lived chains as n_seq * H, which is what launch_stages
// uses for fixed lengths (the only caller); for packed sequences it uses
// H * ceil(T_total / max_len), which this signature cannot see.
// Segments of the scan for B fixed-length sequences of T tokens and H heads
// (1: no scan).  forced > 0 asks for that many; otherwise the scan is used
// when the serial chain would bound the call: long sequences (at least
// kScanMinChunks chunks) and few (sequence, head) chains, with the 2 segs - 1
// walks per chain fitting on the SMs and segs >= 3 (two segments walk the
// same number of chunks in a row as none).  Segments are whole chunks and
// none is empty.
constexpr int kScanMinChunks = 2048, kScanMaxSegs = 8, kScanMaxChains = 64;

int scan_segments(int B, int T, int H, int sms, int forced) {
  const int nc = (T + CH - 1) / CH;
  int segs = forced;
  if (forced <= 0) {
    if (nc < kScanMinChunks || (long long)B * H > kScanMaxChains) return 1;
    segs = std::min(kScanMaxSegs, (sms / (B * H) + 1) / 2);
    if (segs < 3) return 1;
  }
  segs = std::min(std::min(segs, kScanMaxSegs), nc);
  if (segs <= 1) return 1;
  const int per = (nc + segs - 1) / segs;  // chunks per segment
  return (nc + per - 1) / per;
}

bool chunk_fwd_writes_u(int n_seq, int H) {
  int sms = 0;
  return device_sms(&sms) == cudaSuccess && 2 * n_seq * H <= sms;
}

int chunk_fwd_launches(bool packed, int n_seq, int max_len, int H) {
  int sms = 0;
  if (device_sms(&sms) != cudaSuccess) return -1;
  int nc_max = (max_len + CH - 1) / CH;
  if (n_seq <= 0 || nc_max <= 0 || H <= 0) return 0;
  const int segs = packed ? 1 : scan_segments(n_seq, max_len, H, sms, 0);
  if (use_fused(!packed && segs == 1, n_seq * H, nc_max, sms)) return 1;
  int plan = packed ? 1 : 0, chains = n_seq * H, tail = 0;
  if (segs > 1) {  // plan, the walks, combine, second walks
    nc_max = (nc_max + segs - 1) / segs;
    plan = 1;
    chains = n_seq * (2 * segs - 1) * H / 2;
    tail = 2;
  }
  if (!use_overlap(chains, nc_max, sms)) return plan + 2 + tail;
  const int seg = !packed && segs == 1 && ring_records(n_seq, nc_max, H)
                      ? ring_segment_chunks(nc_max, chains) : segment_chunks(nc_max);
  return plan + 2 * ((nc_max + seg - 1) / seg) + tail;
}

namespace {

size_t plan_bytes(int n_seq) { return align_up((size_t)(3 * n_seq + 1) * sizeof(int), 1024); }
// carried states (planes of them: two for a segment scan), then 256 bytes for
// stage 1's counters (finished CTAs, next item)
size_t carry_bytes(int n_seq, int H, int planes = 1) {
  return (size_t)planes * n_seq * H * DP * DP * sizeof(float) + 256;
}
// workspace of a segment scan with segs segments per sequence
size_t scan_workspace_bytes(int B, long long T, int H, int segs) {
  const long long chunks = (long long)B * ((T + CH - 1) / CH);
  return plan_bytes(B * segs) + carry_bytes(B * segs, H, 2) + (size_t)chunks * H * REC_BYTES;
}

}  // namespace

size_t chunk_workspace_bytes(bool packed, int n_seq, long long T_or_total, int H) {
  if (packed) {  // sum of ceil(len / 64) is at most T_total / 64 + N
    const long long chunks = T_or_total / CH + n_seq;
    return plan_bytes(n_seq) + carry_bytes(n_seq, H) + (size_t)chunks * H * REC_BYTES;
  }
  const long long nc = (T_or_total + CH - 1) / CH;
  long long chunks = (long long)n_seq * nc;  // one record per chunk
  // the overlapped schedule keeps the records in a ring of two segments
  int sms = 0;
  if (ring_records(n_seq, (int)nc, H) && device_sms(&sms) == cudaSuccess &&
      use_overlap(n_seq * H, (int)nc, sms))
    chunks = std::min(chunks, (long long)n_seq * 2 * ring_segment_chunks((int)nc, n_seq * H));
  size_t bytes = carry_bytes(n_seq, H) + (size_t)chunks * H * REC_BYTES;
  // shapes that may take the segment scan (which keeps every record): room
  // for its largest form
  if (nc >= kScanMinChunks && (long long)n_seq * H <= kScanMaxChains)
    bytes = std::max(bytes, scan_workspace_bytes(n_seq, T_or_total, H, kScanMaxSegs));
  return bytes;
}

size_t chunk_scan_workspace_bytes(int B, long long T, int H, int segs) {
  if (segs <= 1) return chunk_workspace_bytes(false, B, T, H);
  const int nc = (int)((T + CH - 1) / CH);
  return scan_workspace_bytes(B, T, H, std::min(std::min(segs, kScanMaxSegs), nc));
}

namespace {

// records: per-(chunk, head) records; carry: the state between segments (or
// null, which forces a single segment).
cudaError_t launch_impl(const ChunkProblem& pr, int* plan, float* carry, int* grid_done,
                        uint8_t* records, bool allow_overlap, cudaStream_t stream) {
  const uint64_t d = (uint64_t)pr.d, H = (uint64_t)pr.H;
  const bool packed = pr.cu_seqlens != nullptr;
  if (packed) {
    kda_plan_kernel<<<1, 1024, 0, stream>>>(pr.cu_seqlens, pr.n_seq, pr.T, pr.T_total, plan);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else if (pr.scan_segs > 1) {
    const int B = pr.n_seq / pr.scan_segs;
    kda_segment_plan_kernel<<<(pr.n_seq + 256) / 256, 256, 0, stream>>>(B, pr.T_total / B, pr.T,
                                                                        pr.scan_segs, plan);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int nc_max = (pr.T + CH - 1) / CH;  // T is max_seqlen when packed
  if (nc_max == 0) return cudaSuccess;
  const uint64_t rows = (uint64_t)pr.T_total;
  CUtensorMap tq, tk, tv, tg;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_map_3d_bf16(&tq, pr.q, d, H, rows, d, H * d, 64, 1, 64, sw) ||
      !make_map_3d_bf16(&tk, pr.k, d, H, rows, d, H * d, 64, 1, 64, sw) ||
      !make_map_3d_bf16(&tv, pr.v, d, H, rows, d, H * d, 64, 1, 64, sw) ||
      !make_map_3d_bf16(&tg, pr.log_alpha, d, H, rows, d, H * d, 64, 1, 64, sw))
    return cudaErrorInvalidValue;
  if (pr.d == 128)
    return pr.out_f32 ? launch_stages<128, float>(pr, tq, tk, tv, tg, plan, records, carry,
                                                  grid_done, nc_max, allow_overlap, stream)
                      : launch_stages<128, __nv_bfloat16>(pr, tq, tk, tv, tg, plan, records,
                                                          carry, grid_done, nc_max, allow_overlap, stream);
  return pr.out_f32 ? launch_stages<64, float>(pr, tq, tk, tv, tg, plan, records, carry,
                                               grid_done, nc_max, allow_overlap, stream)
                    : launch_stages<64, __nv_bfloat16>(pr, tq, tk, tv, tg, plan, records,
                                                       carry, grid_done, nc_max, allow_overlap, stream);
}

// The caller's problem has no tokens at all: the final state is the initial state.
cudaError_t copy_initial_state(const ChunkProblem& pr, cudaStream_t stream) {
  if (!pr.final_state) return cudaSuccess;
  const size_t bytes = (size_t)pr.n_seq * pr.H * pr.d * pr.d * sizeof(float);
  if (pr.initial_state)
    return pr.initial_state == pr.final_state
               ? cudaSuccess
               : cudaMemcpyAsync(pr.final_state, pr.initial_state, bytes,
                                 cudaMemcpyDeviceToDevice, stream);
  return cudaMemsetAsync(pr.final_state, 0, bytes, stream);
}

}  // namespace

cudaError_t launch_chunk_fwd(const ChunkProblem& pr_in, void* workspace, cudaStream_t stream) {
  if (pr_in.T_total == 0) return copy_initial_state(pr_in, stream);
  ChunkProblem pr = pr_in;
  int segs = 1;
  if (!pr.cu_seqlens && pr.scan_segs != 0 && pr.scan_segs != 1) {
    int sms = 0;
    cudaError_t e = device_sms(&sms);
    if (e != cudaSuccess) return e;
    segs = scan_segments(pr.n_seq, pr.T, pr.H, sms, pr.scan_segs > 0 ? pr.scan_segs : 0);
  }
  if (segs > 1) {  // the segments become the sequences of the work list
    const int nc = (pr.T + CH - 1) / CH, per = (nc + segs - 1) / segs;
    pr.n_seq *= segs;
    pr.T = per * CH;
  }
  pr.scan_segs = segs;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* plan = nullptr;
  if (pr.cu_seqlens || segs > 1) {
    plan = reinterpret_cast<int*>(ws);
    ws += plan_bytes(pr.n_seq);
  }
  const int planes = segs > 1 ? 2 : 1;
  float* carry = reinterpret_cast<float*>(ws);
  int* grid_done = reinterpret_cast<int*>(ws + carry_bytes(pr.n_seq, pr.H, planes) - 256);
  ws += carry_bytes(pr.n_seq, pr.H, planes);
  return launch_impl(pr, plan, carry, grid_done, ws, true, stream);
}

// ---- allocation-free variant --------------------------------------------
// Scratch for kda_chunk_fwd_noalloc: a fixed 64 MiB device array that every
// GPU loading this library holds until the process exits.  It holds up to
// 1008 per-(chunk, head) records.  All calls share it and nothing in it has
// to start at zero (every record is written before it is read); calls whose
// work overlaps on the GPU race on it.
namespace {
constexpr size_t kNoAllocBytes = (size_t)64 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];
}  // namespace

size_t noalloc_max_records() { return kNoAllocBytes / REC_BYTES; }

cudaError_t launch_chunk_fwd_noalloc(const ChunkProblem& pr, cudaStream_t stream) {
  // The array's device address on the current device.  In host code the
  // symbol is only a host-side stand-in, so the address is looked up with
  // the device current, on every call: the lookup allocates nothing, and a
  // fresh lookup stays right after a device reset reloads the module.
  void* scratch = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (pr.T_total == 0) return copy_initial_state(pr, stream);
  // one segment (no carried state, no internal streams), records only
  return launch_impl(pr, nullptr, nullptr, nullptr, static_cast<uint8_t*>(scratch), false, stream);
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
