// Test-only probes of the building blocks in umma.cuh.  They run one
// tcgen05.mma sequence, or one TMA tile load, on operands placed in shared
// memory by the same layout functions the KDA kernels use, and hand the raw
// result back so a test can compare it with a host matmul / slice.  Not part
// of the product library (built into libkda_probe.so).
#include <cuda_runtime.h>

#include "../../include/kda_probe.h"
#include "tma_host.h"
#include "umma.cuh"

using namespace kda;

namespace {

struct ProbeArgs {
  int M, N, K, NB;
  int a_mn, a_sw, a_mn_blocks_contig;
  int b_mn, b_sw, b_mn_blocks_contig;
  int b_row0, neg_a, n_accum;
  int tf32;  // operands are fp32, MMA kind::tf32
  int a_tmem;  // A is written to tensor memory (bf16 pairs per column) and read from there
};

constexpr int kProbeSmem = 1024 + 32 * 1024 + 64 * 1024 + 1024;

__host__ __device__ OperandLayout probe_layout(uint32_t base, int rows, int K, int mn, int sw,
                                               int blocks_contig, uint32_t esize) {
  OperandLayout L;
  L.base = base;
  L.esize = esize;
  L.sw = (uint32_t)sw;
  L.mn_major = mn != 0;
  const uint32_t S = swizzle_bytes(L.sw);
  const uint32_t W = S / esize;
  if (!L.mn_major) {
    L.sbo = 8 * S;
    L.kb_stride = (uint32_t)rows * S;
    L.lbo = 0;
  } else if (!blocks_contig) {  // the K groups of one MN block are contiguous
    L.sbo = 8 * S;
    L.lbo = (uint32_t)K * S;  // K rows of S bytes per MN block
    L.kb_stride = 0;
  } else {  // the MN blocks of one K group are contiguous
    L.lbo = 8 * S;
    L.sbo = ((uint32_t)rows / W) * 8 * S;
    L.kb_stride = 0;
  }
  return L;
}

__global__ void __launch_bounds__(128) probe_umma_kernel(const __nv_bfloat16* __restrict__ A,
                                                         const __nv_bfloat16* __restrict__ B,
                                                         float* __restrict__ D, ProbeArgs p,
                                                         int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t a_base = (raw + 1023u) & ~1023u;
  const uint32_t b_base = a_base + 32 * 1024;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  const uint32_t es = p.tf32 ? 4u : 2u;
  const OperandLayout LA = probe_layout(a_base, p.M, p.K, p.a_mn, p.a_sw, p.a_mn_blocks_contig, es);
  const OperandLayout LB = probe_layout(b_base, p.NB, p.K, p.b_mn, p.b_sw, p.b_mn_blocks_contig, es);
  // zero both regions, then scatter the logical matrices into them
  for (uint32_t off = tid * 16; off < 96 * 1024; off += 128 * 16) st_shared_v4(a_base + off, 0, 0, 0, 0);
  __syncthreads();
  for (int idx = tid; idx < p.M * p.K; idx += 128) {
    const int r = idx / p.K, k = idx % p.K;
    if (p.tf32)
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(layout_addr(LA, r, k)), "f"(__bfloat162float(A[idx])));
    else
      st_shared_u16(layout_addr(LA, r, k), __bfloat16_as_ushort(A[idx]));
  }
  for (int idx = tid; idx < p.NB * p.K; idx += 128) {
    const int r = idx / p.K, k = idx % p.K;
    if (p.tf32)
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(layout_addr(LB, r, k)), "f"(__bfloat162float(B[idx])));
    else
      st_shared_u16(layout_addr(LB, r, k), __bfloat16_as_ushort(B[idx]));
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = tmem_base_s;
  constexpr uint32_t kATmemCol = 256;
  if (p.a_tmem) {  // thread (warp, lane) writes row 32 warp + lane of A: K / 2 packed columns
    const int m = 32 * warp + lane;
    for (int c0 = 0; c0 < p.K / 2; c0 += 16) {
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int kk = 2 * (c0 + i);
        const uint32_t lo = m < p.M ? __bfloat16_as_ushort(A[m * p.K + kk]) : 0u;
        const uint32_t hi = m < p.M ? __bfloat16_as_ushort(A[m * p.K + kk + 1]) : 0u;
        x[i] = __uint_as_float(lo | (hi << 16));
      }
      tmem_st16(tmem_addr(tbase, 32 * warp, kATmemCol + c0), x);
    }
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
  }

  if (tid == 0) {
    if (p.tf32) {
      const uint32_t idesc = make_idesc_tf32(p.M, p.N, p.a_mn != 0, p.b_mn != 0);
      for (int rep = 0; rep < p.n_accum; ++rep)
        for (int k0 = 0; k0 < p.K; k0 += 8)
          umma_tf32(tbase, layout_desc(LA, 0, k0), layout_desc(LB, p.b_row0, k0), idesc,
                    (rep > 0 || k0 > 0) ? 1u : 0u);
    } else if (p.a_tmem) {
      const uint32_t idesc = make_idesc_bf16(p.M, p.N, false, p.b_mn != 0, p.neg_a != 0);
      for (int rep = 0; rep < p.n_accum; ++rep)
        for (int k0 = 0; k0 < p.K; k0 += 16)
          umma_f16_ta(tbase, tbase + kATmemCol + k0 / 2, layout_desc(LB, p.b_row0, k0), idesc,
                      (rep > 0 || k0 > 0) ? 1u : 0u);
    } else {
      const uint32_t idesc = make_idesc_bf16(p.M, p.N, p.a_mn != 0, p.b_mn != 0, p.neg_a != 0);
      for (int rep = 0; rep < p.n_accum; ++rep)
        for (int k0 = 0; k0 < p.K; k0 += 16)
          umma_bf16(tbase, layout_desc(LA, 0, k0), layout_desc(LB, p.b_row0, k0), idesc,
                    (rep > 0 || k0 > 0) ? 1u : 0u);
    }
    umma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0);
  if (!ok) {
    // the MMAs may still be writing TMEM: give them one more bounded wait
    // before the columns are freed below
    if (lane == 0) atomicExch(status, 6);
    mbar_wait(&bar, 0, 100000000ull);
  }
  tc_fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < p.N; c0 += 16) {
      float v[16];
      tmem_ld16(tmem_addr(tbase, 32 * warp, c0), v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) D[(size_t)(32 * warp + lane) * p.N + c0 + i] = v[i];
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

__global__ void __launch_bounds__(128) probe_tma_kernel(const __grid_constant__ CUtensorMap map,
                                                        __nv_bfloat16* __restrict__ out, int d,
                                                        int h, int t0, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t bar;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int nblk = d / 64;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)nblk * 64 * 64 * 2);
    for (int b = 0; b < nblk; ++b)
      tma_load_3d(base_ptr + b * 8192, &map, &bar, b * 64, h, t0);
  }
  if (!mbar_wait(&bar, 0)) {
    // the tile may still be landing in this CTA's shared memory: one more
    // bounded wait before the CTA exits
    if (threadIdx.x == 0) atomicExch(status, 6);
    mbar_wait(&bar, 0, 100000000ull);
    return;
  }
  // read back through the K-major SW128 layout: row = token, k = channel
  OperandLayout L;
  L.base = base;
  L.sw = SW_128;
  L.mn_major = false;
  L.sbo = 1024;
  L.kb_stride = 8192;
  L.lbo = 0;
  for (int idx = threadIdx.x; idx < 64 * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    out[idx] = __ushort_as_bfloat16(ld_shared_u16(layout_addr(L, r, c)));
  }
}

// A wait that runs out on purpose: TMEM is allocated, an mbarrier is set up
// that nothing ever arrives on, and every thread waits on it through the
// same bounded wait the KDA kernels use, with a limit of limit_ns.  The
// wait gives up, the kernel records KDA_ERR_TIMEOUT (6) in *status, frees
// its TMEM and returns, leaving the context usable.
__global__ void __launch_bounds__(128) probe_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, 32);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = tmem_base_s;
  const bool ok = mbar_wait(&bar, 0, limit_ns);
  if (!ok && threadIdx.x == 0) atomicExch(status, 6);
  if (ok && threadIdx.x == 0) atomicExch(status, -1);  // cannot happen: nothing arrives
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 32);
}

}  // namespace

extern "C" KDA_API int kda_probe_wait_timeout(int limit_us, int* status, cudaStream_t stream) {
  if (limit_us <= 0 || limit_us > 100000 || !status) return 1;
  probe_timeout_kernel<<<1, 128, 0, stream>>>((uint64_t)limit_us * 1000ull, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

extern "C" KDA_API int kda_probe_umma(const void* A, const void* B, float* D, int M, int N, int K, int NB,
                              int a_mn, int a_sw, int a_mn_blocks_contig, int b_mn, int b_sw,
                              int b_mn_blocks_contig, int b_row0, int neg_a, int n_accum,
                              int tf32, int* status, cudaStream_t stream) {
  return kda_probe_umma_ta(A, B, D, M, N, K, NB, a_mn, a_sw, a_mn_blocks_contig, b_mn, b_sw,
                           b_mn_blocks_contig, b_row0, neg_a, n_accum, tf32, 0, status, stream);
}

extern "C" KDA_API int kda_probe_umma_ta(const void* A, const void* B, float* D, int M, int N,
                                         int K, int NB, int a_mn, int a_sw,
                                         int a_mn_blocks_contig, int b_mn, int b_sw,
                                         int b_mn_blocks_contig, int b_row0, int neg_a,
                                         int n_accum, int tf32, int a_tmem, int* status,
                                         cudaStream_t stream) {
  if (a_tmem && (M != 128 || tf32 || a_mn || K > 128)) return 1;
  if (!(M == 64 || M == 128) || N < 16 || N > 256 || N % 16 || K % 16 || K > 128 || K < 16)
    return 1;
  if (NB < b_row0 + N || NB > 256 || (a_mn && M % 64) || n_accum < 1) return 1;
  if (tf32 && (neg_a || (size_t)NB * K * 4 > 64 * 1024 || (size_t)M * K * 4 > 32 * 1024)) return 1;
  ProbeArgs p{M, N, K, NB, a_mn, a_sw, a_mn_blocks_contig, b_mn, b_sw, b_mn_blocks_contig,
              b_row0, neg_a, n_accum, tf32, a_tmem};
  if (cudaFuncSetAttribute(probe_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kProbeSmem) != cudaSuccess)
    return 4;
  probe_umma_kernel<<<1, 128, kProbeSmem, stream>>>(static_cast<const __nv_bfloat16*>(A),
                                                    static_cast<const __nv_bfloat16*>(B), D, p,
                                                    status);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

extern "C" KDA_API int kda_probe_tma(const void* src, void* out, int T, int H, int d, int h, int t0,
                             int* status, cudaStream_t stream) {
  if (!(d == 64 || d == 128) || h < 0 || h >= H) return 1;
  CUtensorMap map;
  if (!make_map_3d_bf16(&map, src, (uint64_t)d, (uint64_t)H, (uint64_t)T, (uint64_t)d,
                        (uint64_t)H * d, 64, 1, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return 4;
  const int smem = 1024 + 16384;
  if (cudaFuncSetAttribute(probe_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 4;
  probe_tma_kernel<<<1, 128, smem, stream>>>(map, static_cast<__nv_bfloat16*>(out), d, h, t0,
                                             status);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
