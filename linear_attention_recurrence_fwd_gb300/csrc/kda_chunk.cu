// Chunked KDA prefill (placeholder until the tcgen05 kernel lands).
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

static __device__ int g_chunk_status = 0;

cudaError_t launch_chunk_fwd(const ChunkProblem&, cudaStream_t) { return cudaErrorNotYetImplemented; }

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
