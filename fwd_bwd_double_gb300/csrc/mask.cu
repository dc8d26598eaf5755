// Document (segment) mask bounds.  "FlashBoB: second-order attention", section "When
// FlashBoB changes the engineering plan", lists flexible masks among the next extensions;
// the document mask is the one packed training batches use: query i sees key j iff
// j <= i and both carry the same segment id.  With the ids of a batch row non-decreasing
// (each document one run), row i's visible keys are the range lo(i) <= j <= i and key j's
// rows the range j <= i <= hi(j), where lo(i) is the first and hi(j) the last index of the
// token's run.  This launch computes both per token, once per batch of sequences; every
// attention call then reads two integers per row or key instead of searching.
#include <cuda_runtime.h>

#include "internal.h"

namespace fbd {
namespace {

// One thread per token: lo = first index in [0, i] whose id equals seg[i] (a lower bound
// in the non-decreasing ids), hi = last index in [i, N - 1] with that id.  Both stay in
// [0, i] and [i, N - 1] for any ids, so the row always keeps its own key.
__global__ void __launch_bounds__(256) segment_bounds_kernel(const int* __restrict__ seg, int* __restrict__ lo,
                                                             int* __restrict__ hi, int64_t N, int64_t total) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int64_t b = t / N, i = t - b * N;
  const int* row = seg + b * N;
  const int v = row[i];
  int64_t a = 0, z = i;  // smallest index in [a, z] with row[index] >= v (z qualifies)
  while (a < z) {
    const int64_t m = a + ((z - a) >> 1);
    if (row[m] >= v) z = m; else a = m + 1;
  }
  lo[t] = static_cast<int>(a);
  a = i;
  z = N - 1;  // largest index in [a, z] with row[index] <= v (a qualifies)
  while (a < z) {
    const int64_t m = a + ((z - a + 1) >> 1);
    if (row[m] <= v) a = m; else z = m - 1;
  }
  hi[t] = static_cast<int>(a);
}

}  // namespace

cudaError_t segment_bounds(int64_t B, int64_t N, const int* seg, int* lo, int* hi, cudaStream_t st) {
  const int64_t total = B * N;
  if (total == 0) return cudaSuccess;
  segment_bounds_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(seg, lo, hi, N, total);
  return cudaGetLastError();
}

}  // namespace fbd
