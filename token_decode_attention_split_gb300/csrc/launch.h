// Internal launch interface between the C ABI (api.cu) and the per-variant kernel translation
// units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode_kernel.cuh"
#include "host_api.h"

namespace da {

struct Launch {
    CUtensorMap tm_k;   // unused by the sparse kernels
    CUtensorMap tm_v;
    Params p;
    int grid;
    int threads;        // block size of the variant
    cudaStream_t stream;
};

cudaError_t launch_dense(int D, int GP, const Launch& L);
// Paged units of one KV head (kh == 1).
cudaError_t launch_paged_single(int D, int GP, const Launch& L);
// Paged units of kh > 1 KV heads.  warp_head: each consumer warp holds only the query columns of
// the KV head its rows belong to (pages of >= 16 rows, <= 8 columns per KV head, GP == 16).
cudaError_t launch_paged_multi(int D, int GP, bool warp_head, const Launch& L);
cudaError_t launch_sparse(int D, int GP, const Launch& L);
// Sparse units of 33..64 query heads (head dim 64 or 128) on the tcgen05 kernel (sparse_tc.cu):
// block size and launch; its chunks are kSparseChunkUnit entries like the mma.sync kernel's.
int sparse_tc_threads();
cudaError_t launch_sparse_tc(int D, const Launch& L);

// One 32-thread block whose bounded wait on a never-completed barrier times out after limit_ns
// and records kErrWaitCheck in *err.
cudaError_t launch_wait_check(unsigned* err, uint64_t limit_ns, cudaStream_t stream);

// Opts the kernel into `smem` bytes of dynamic shared memory on the current device (once per
// kernel and CUDA context), then launches it with L.threads threads per block.
cudaError_t launch_kernel(const void* kernel, int smem, const Launch& L);


}  // namespace da
