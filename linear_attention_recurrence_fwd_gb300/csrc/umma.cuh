// Blackwell (sm_100 family) building blocks written as inline PTX:
// shared-memory matrix descriptors and canonical operand layouts for
// tcgen05.mma, TMEM allocation / load / store, mbarriers with bounded waits,
// and TMA tile loads.  Everything here is layout bookkeeping; the KDA
// arithmetic lives in the kernels that include this file.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace kda {

// ---------------------------------------------------------------- addresses
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete.  Gives up after
// `limit_ns` of wall time (read from %globaltimer) and returns false, so a
// lost arrival can never hang the GPU: the caller records a timeout status
// and unwinds.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- fences
// Generic-proxy smem writes -> visible to the async proxy (tensor core, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM
// Allocation is warp-wide; the TMEM base address is written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// TMEM address: lane in bits [31:16], column in bits [15:0].
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  return __uint_as_float(r);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- UMMA
// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bit 46, and the
// swizzle mode in bits [61,64).
enum Swizzle : uint32_t { SW_NONE = 0, SW_128 = 2, SW_64 = 4, SW_32 = 6 };

__host__ __device__ constexpr uint32_t swizzle_bytes(uint32_t sw) {
  return sw == SW_128 ? 128u : sw == SW_64 ? 64u : sw == SW_32 ? 32u : 16u;
}

__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t sw) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)(sw & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with an fp32 accumulator; A and B
// are both bf16 (fp16 = false) or both fp16 (fp16 = true).
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn_major, bool b_mn_major,
                                                  bool negate_a = false, bool fp16 = false) {
  return (1u << 4)                               // D format: f32
         | ((fp16 ? 0u : 1u) << 7)               // A format: 0 = f16, 1 = bf16
         | ((fp16 ? 0u : 1u) << 10)              // B format
         | ((negate_a ? 1u : 0u) << 13)          // negate A
         | ((a_mn_major ? 1u : 0u) << 15)        // A major: 0 = K, 1 = MN
         | ((b_mn_major ? 1u : 0u) << 16)        // B major
         | ((uint32_t)(N >> 3) << 17)            // N / 8
         | ((uint32_t)(M >> 4) << 24);           // M / 16
}

__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool a_mn_major,
                                                       bool b_mn_major, bool negate_a = false) {
  return make_idesc(M, N, a_mn_major, b_mn_major, negate_a, false);
}

// kind::tf32: fp32 operands read as tf32 (10-bit mantissa, fp32 range), K = 8 per MMA.
__host__ __device__ constexpr uint32_t make_idesc_tf32(int M, int N, bool a_mn_major,
                                                       bool b_mn_major) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (A and B both bf16 or both
// fp16), A read from tensor memory: row m of A in lane m, two consecutive
// K elements per 32-bit column (the lower half the even one).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ------------------------------------------------ canonical operand layouts
// An operand tile of R rows (its M or N extent) by K columns of bf16.
//
// K-major (K contiguous), swizzle width S bytes: K is cut into blocks of S/2
// elements; block kb is a dense R x S-byte region at kb * kb_stride; inside
// it rows sit S bytes apart and 8-row groups SBO = 8*S bytes apart.  The XOR
// swizzle acts on absolute smem address bits, so regions are aligned to 8*S.
//
// MN-major (rows contiguous), swizzle width S bytes: an atom is 8 K-rows of
// S bytes (S/2 consecutive MN elements each).  MN-blocks of S/2 elements
// are LBO apart, groups of 8 K-rows are SBO apart.
struct OperandLayout {
  uint32_t base;       // smem byte address of the tile (aligned to 8*S)
  uint32_t esize = 2;  // element bytes (2: bf16/fp16, 4: tf32)
  uint32_t sw;         // Swizzle code
  bool mn_major;
  uint32_t lbo;        // MN-major: stride between MN blocks
  uint32_t sbo;        // stride between 8-row (K-major) / 8-K (MN-major) groups
  uint32_t kb_stride;  // K-major: stride between K blocks of S/2 elements
};

// Byte offset (relative to base, before swizzle) of element (row, k).
__host__ __device__ __forceinline__ uint32_t layout_offset(const OperandLayout& L, uint32_t row,
                                                           uint32_t k) {
  const uint32_t S = swizzle_bytes(L.sw);
  const uint32_t W = S / L.esize;  // elements per atom row
  if (!L.mn_major) {
    return (k / W) * L.kb_stride + (row / 8) * L.sbo + (row % 8) * S + (k % W) * L.esize;
  }
  return (row / W) * L.lbo + (k / 8) * L.sbo + (k % 8) * S + (row % W) * L.esize;
}

// Apply the XOR swizzle (16-byte chunk index ^= 128-byte line index, masked
// to the swizzle width) to an absolute smem byte address.
__host__ __device__ __forceinline__ uint32_t swizzle_addr(uint32_t addr, uint32_t sw) {
  const uint32_t bits = sw == SW_128 ? 3u : sw == SW_64 ? 2u : sw == SW_32 ? 1u : 0u;
  const uint32_t mask = (1u << bits) - 1u;
  return addr ^ (((addr >> 7) & mask) << 4);
}

__host__ __device__ __forceinline__ uint32_t layout_addr(const OperandLayout& L, uint32_t row,
                                                         uint32_t k) {
  return swizzle_addr(L.base + layout_offset(L, row, k), L.sw);
}

// Descriptor for the K slice starting at k0 (16 wide for 16-bit types, 8 for tf32), rows
// starting at row0 (row0 % 8 == 0 for K-major; MN-major row0 may point
// inside an atom row, which moves the start address by row0*2 bytes).
__device__ __forceinline__ uint64_t layout_desc(const OperandLayout& L, uint32_t row0,
                                                uint32_t k0) {
  const uint32_t start = L.base + layout_offset(L, row0, k0);
  return make_sdesc(start, L.mn_major ? L.lbo : 16u, L.sbo, L.sw);
}

// Advance a 128B-swizzled 16-bit operand descriptor (built for K = 0) to the
// K slice at k0.  MN-major: k0 / 8 groups of 8 K-rows, 1024 bytes apart;
// K-major: k0 / 64 K-blocks kb_stride apart, plus 2 bytes per element inside
// the 128-byte atom row.  With k0 a compile-time constant this folds to one
// 64-bit add on the start-address field (addresses stay below 256 KiB).
__device__ __forceinline__ uint64_t desc_adv(uint64_t d, int k0, bool mn_major,
                                             uint32_t kb_stride = 0) {
  const uint32_t bytes = mn_major ? (uint32_t)(k0 >> 3) * 1024u
                                  : (uint32_t)(k0 >> 6) * kb_stride + (uint32_t)(k0 & 63) * 2u;
  return d + (bytes >> 4);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Untiled bulk copies (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_global, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(src_global)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst_global, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst_global)),
               "r"(src_smem), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk store has finished (reads and writes).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_reads() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed bulk group but the most recent one is done reading shared memory.
__device__ __forceinline__ void bulk_wait_reads_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}

}  // namespace kda
