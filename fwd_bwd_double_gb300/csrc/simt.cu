// The GProj projected-dS diagnostic export (bf16 inputs), on the CUDA cores: it writes
// the whole N x N matrix dS~ = bf16(dS) - rho bf16(P) per (batch, head) for inspection
// ("FlashAttention bf16 gradient and GProj", "How the zero sum turns into a false
// gradient"), so it is a small-N test and teaching aid, not a hot-path kernel.  Every
// forward, backward and BoB runs on the tensor cores (tc_*.cu).
//
// One warp per query row; the lanes hold d/32 consecutive elements of the row's vectors
// (coalesced row reads), dot products are warp butterfly reductions.  P is recomputed
// from lse ("Backward pass: recompute instead of store").
#include <cuda_bf16.h>
#include <math_constants.h>

#include <type_traits>

#include "internal.h"

namespace fbd {
namespace {

constexpr int kWarps = 8;       // rows per CTA
constexpr int kThreads = kWarps * 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }


__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

template <int V, typename T>
__device__ __forceinline__ void load_vec(const T* __restrict__ row, int lane, float (&v)[V]) {
#pragma unroll
  for (int t = 0; t < V; ++t) v[t] = to_f(row[lane * V + t]);
}

template <int K>
__device__ __forceinline__ void warp_sum(float (&x)[K]) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int k = 0; k < K; ++k) x[k] += __shfl_xor_sync(kFull, x[k], off);
}

template <int V>
__device__ __forceinline__ float dot(const float (&x)[V], const float (&y)[V]) {
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < V; ++t) s = fmaf(x[t], y[t], s);
  return s;
}


// Slice/row-block decode of the 1-D grid: blockIdx.x = blk * BH + bh, heaviest
// causal blocks (largest blk for row passes) first.
struct Tile {
  int64_t bh, blk;
};
__device__ __forceinline__ Tile decode(int64_t BH, int64_t nblk, bool heavy_last_rows) {
  const int64_t x = blockIdx.x;
  Tile t;
  t.bh = x % BH;
  const int64_t k = x / BH;
  t.blk = heavy_last_rows ? (nblk - 1 - k) : k;
  return t;
}

// ------------------------------------------- GProj projected dS (diagnostic)
// One warp per row: sweep 1 accumulates r = sum bf16(dS) and sum bf16(P);
// sweep 2 writes dS~ = bf16(dS) - rho bf16(P) for every visible key (0 for j > i
// under the causal mask).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) projected_dS_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                                const T* __restrict__ Vt, const T* __restrict__ O,
                                                                const T* __restrict__ dO,
                                                                const float* __restrict__ lse,
                                                                float* __restrict__ out, int64_t N, int64_t BH,
                                                                float scale, int causal, Band bd, int64_t G) {
  constexpr int V = D / 32;
  const int64_t nblk = (N + kWarps - 1) / kWarps;
  const Tile tl = decode(BH, nblk, true);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t i = tl.blk * kWarps + warp;
  if (i >= N) return;
  const size_t base = static_cast<size_t>(tl.bh) * N * D;
  const size_t kvbase = static_cast<size_t>(tl.bh / G) * N * D;
  float q[V], g[V], o[V];
  load_vec(Q + base + i * D, lane, q);
  load_vec(dO + base + i * D, lane, g);
  load_vec(O + base + i * D, lane, o);
  float x0[1] = {dot(g, o)};
  warp_sum(x0);
  const float Di = x0[0], Li = lse[tl.bh * N + i];
  const int64_t lo_i = causal ? bd.row_lo(tl.bh, i) : 0;  // this row's first visible key
  float r = 0.f, sp = 0.f;
  for (int pass = 0; pass < 2; ++pass) {
    const float rho = r / sp;
    for (int64_t j = 0; j < N; ++j) {
      float* dst = out + (static_cast<size_t>(tl.bh) * N + i) * N + j;
      if (causal && (j > i || j < lo_i)) {
        if (pass == 1 && lane == 0) *dst = 0.f;
        continue;
      }
      float kv[V], vv[V];
      load_vec(K + kvbase + j * D, lane, kv);
      load_vec(Vt + kvbase + j * D, lane, vv);
      float x[2] = {dot(q, kv), dot(g, vv)};
      warp_sum(x);
      const float p = expf(x[0] * scale - Li);
      const float dsh = bf16r(p * (x[1] - Di)), ph = bf16r(p);
      if (pass == 0) {
        r += dsh;
        sp += ph;
      } else if (lane == 0) {
        *dst = dsh - rho * ph;
      }
    }
  }
}

inline unsigned grid_for(const Problem& p) {
  return static_cast<unsigned>(((p.N + kWarps - 1) / kWarps) * p.BH);
}

}  // namespace

// Head dimensions the CUDA-core kernels are built for (a warp's lanes hold d/32
// elements each).  Returns false for any other d.
template <typename F>
bool with_head_dim(int64_t d, F&& f) {
  switch (d) {
    case 32: f(std::integral_constant<int, 32>{}); return true;
    case 64: f(std::integral_constant<int, 64>{}); return true;
    case 96: f(std::integral_constant<int, 96>{}); return true;
    case 128: f(std::integral_constant<int, 128>{}); return true;
    case 256: f(std::integral_constant<int, 256>{}); return true;
  }
  return false;
}

cudaError_t simt_projected_dS(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* lse, float* dS, cudaStream_t st) {
  using T = __nv_bfloat16;
  cudaError_t e = cudaErrorInvalidValue;
  with_head_dim(p.d, [&](auto dd) {
    projected_dS_kernel<T, dd()><<<grid_for(p), kThreads, 0, st>>>(
        static_cast<const T*>(Q), static_cast<const T*>(K), static_cast<const T*>(V), static_cast<const T*>(O),
        static_cast<const T*>(dO), lse, dS, p.N, p.BH, p.scale, p.causal, make_band(p, eff_window(p), false), p.group);
    e = cudaGetLastError();
  });
  return e;
}

}  // namespace fbd
