// Validation of a packed batch's sequence boundaries on the device.
//
// The RoPE kernels read cu_seqlens on the GPU so the host never waits for it
// ("Unsloth und NVIDIA optimieren LLM-Training um zusätzliche 25%",
// lumeric.app, item (1): the packed-sequence metadata is kept where the
// kernels use it instead of synchronising the host).  A malformed batch can
// then only give wrong positions, silently.  This kernel checks the
// boundaries where they live and writes what it found to a caller-owned
// device word; the checked RoPE entry points read that word and leave q and k
// untouched when it is non-zero.  Nothing traps or faults.
//
// One CTA: thread i tests cu[i] <= cu[i+1] for i = tid, tid + 1024, ...;
// thread 0 tests cu[0] == 0 and cu[B] == T.  The bits are OR-ed across the
// CTA and thread 0 overwrites the word, so it needs no clearing between
// batches.
#include "common.cuh"
#include "ftk.h"
#include "launch.h"

namespace ftk {

namespace {

constexpr int kCheckThreads = 1024;

__global__ void __launch_bounds__(kCheckThreads)
check_seqlens_kernel(const int32_t *__restrict__ cu, int32_t B, int64_t T,
                     uint32_t *__restrict__ status) {
  pdl_wait();  // cu may come from the preceding kernel; a preceding RoPE may read status
  pdl_trigger();
  uint32_t bad = 0;
  for (int64_t i = threadIdx.x; i < (int64_t)B; i += kCheckThreads)
    if (__ldg(cu + i + 1) < __ldg(cu + i)) bad |= FTK_SEQLENS_DECREASING;
  if (threadIdx.x == 0) {
    if (__ldg(cu) != 0) bad |= FTK_SEQLENS_BAD_START;
    if ((int64_t)__ldg(cu + B) != T) bad |= FTK_SEQLENS_BAD_END;
  }
  // OR of the bits over the CTA, two at a time through the predicate form
  const int dec = __syncthreads_or((bad & FTK_SEQLENS_DECREASING) != 0);
  if (threadIdx.x == 0)
    *status = (bad & (FTK_SEQLENS_BAD_START | FTK_SEQLENS_BAD_END)) |
              (dec ? FTK_SEQLENS_DECREASING : 0u);
}

}  // namespace

cudaError_t launch_check_seqlens(const int32_t *cu, int32_t B, int64_t T, uint32_t *status,
                                 cudaStream_t s) {
  cudaError_t e = launch_pdl(check_seqlens_kernel, dim3(1), dim3(kCheckThreads), 0, s, cu, B, T,
                             status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ftk
