// CUDA-core path: the backward and BoB in fp32 arithmetic for the bf16 cases that
// have no tensor-core kernel (GProj at d = 256: bf16 is widened on load and rounded
// once on store; the bf16 rounding of dS and P is emulated), and the GProj
// projected-dS diagnostic export.  float32 inputs run on the tf32 tensor-core kernels
// (tc_f32.cu) at every head dim.
//
// Work split: one warp per query row (row passes) or per key (column passes);
// a warp's 32 lanes each hold d/32 consecutive elements of the row's vectors, so
// every global row read is one coalesced 128/256/512-byte access.  The CTA's 8
// warps share a shared-memory staging tile of 32 partner rows (keys for row
// passes, queries for column passes), converted to fp32 once.  Dot products are
// warp butterfly reductions; all lanes then hold the same value, so the softmax
// bookkeeping is warp-uniform.
//
// These kernels follow the same decomposition as the tensor-core path:
//   backward: recompute P from lse ("Backward pass: recompute instead of store");
//   BoB: row pass with the two scalar states, column pass re-reading them
//        ("FlashBoB: second-order attention", "Two scalar states replace
//        quadratic tensors").
#include <cuda_bf16.h>
#include <math_constants.h>

#include <type_traits>

#include "internal.h"

namespace fbd {
namespace {

constexpr int kWarps = 8;       // rows (or keys) per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 32;       // partner rows staged per step
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t lmax(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

template <int V, typename T>
__device__ __forceinline__ void load_vec(const T* __restrict__ row, int lane, float (&v)[V]) {
#pragma unroll
  for (int t = 0; t < V; ++t) v[t] = to_f(row[lane * V + t]);
}
template <int V, typename T>
__device__ __forceinline__ void store_vec(T* __restrict__ row, int lane, const float (&v)[V]) {
#pragma unroll
  for (int t = 0; t < V; ++t) row[lane * V + t] = from_f<T>(v[t]);
}
template <int V>
__device__ __forceinline__ void load_smem(const float* __restrict__ row, int lane, float (&v)[V]) {
#pragma unroll
  for (int t = 0; t < V; ++t) v[t] = row[lane * V + t];
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

// Stage rows [r0, r0 + kTile) of a [N, D] slice into shared memory as fp32 (0 past N).
template <typename T, int D>
__device__ __forceinline__ void stage(float* __restrict__ dst, const T* __restrict__ src, int64_t r0, int64_t N) {
  for (int e = threadIdx.x; e < kTile * D; e += kThreads) {
    const int r = e / D;
    const int64_t gr = r0 + r;
    dst[e] = gr < N ? to_f(src[gr * D + (e % D)]) : 0.f;
  }
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

// --------------------------------------------------------- backward, rows
// dQ and the row statistics (lse, D, rho, 0).  GPROJ rounds dS and P to bf16 as
// the bf16 tensor-core path does and applies the GProj projection.
template <typename T, int D, bool GPROJ>
__global__ void __launch_bounds__(kThreads) bwd_row_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                           const T* __restrict__ Vt, const T* __restrict__ O,
                                                           const T* __restrict__ dO, const float* __restrict__ lse,
                                                           T* __restrict__ dQ, float4* __restrict__ ws, int64_t N,
                                                           int64_t BH, float scale, int causal, Band bd, int64_t G) {
  constexpr int V = D / 32;
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = sm + kTile * D;
  const int64_t nblk = (N + kWarps - 1) / kWarps;
  const Tile tl = decode(BH, nblk, true);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t row0 = tl.blk * kWarps, i = row0 + warp;
  const bool live = i < N;
  const size_t base = static_cast<size_t>(tl.bh) * N * D;
  const size_t kvbase = static_cast<size_t>(tl.bh / G) * N * D;
  float q[V], g[V], acc[V], pk[V];
  float Di = 0.f, Li = 0.f, r = 0.f, sp = 0.f;
#pragma unroll
  for (int t = 0; t < V; ++t) acc[t] = pk[t] = 0.f;
  if (live) {
    float o[V];
    load_vec(Q + base + i * D, lane, q);
    load_vec(dO + base + i * D, lane, g);
    load_vec(O + base + i * D, lane, o);
    float x[1] = {dot(g, o)};
    warp_sum(x);
    Di = x[0];
    Li = lse[tl.bh * N + i];
  }
  const int64_t last = causal ? min(row0 + kWarps, N) - 1 : N - 1;  // last key any row of the block sees
  // bd: the banded causal mask (row i sees the keys bd.row_lo(i) <= j <= i)
  const int64_t first = causal ? (bd.row_lo(tl.bh, row0) / kTile) * kTile : 0;  // first key tile any row sees
  const int64_t lo_i = causal ? bd.row_lo(tl.bh, i) : 0;  // this row's first visible key
  for (int64_t k0 = first; k0 <= last; k0 += kTile) {
    __syncthreads();
    stage<T, D>(Ks, K + kvbase, k0, N);
    stage<T, D>(Vs, Vt + kvbase, k0, N);
    __syncthreads();
    if (!live) continue;
    const int jn = static_cast<int>(lmin(kTile, (causal ? i + 1 : N) - k0));
    const int jb = causal ? static_cast<int>(lmin(kTile, lmax(0, lo_i - k0))) : 0;  // below the row's band
    for (int jj = jb; jj < jn; ++jj) {
      float kv[V], vv[V];
      load_smem(Ks + jj * D, lane, kv);
      load_smem(Vs + jj * D, lane, vv);
      float x[2] = {dot(q, kv), dot(g, vv)};
      warp_sum(x);
      const float p = expf(x[0] * scale - Li);
      const float ds = p * (x[1] - Di);
      if constexpr (GPROJ) {
        const float dsh = bf16r(ds), ph = bf16r(p);
        r += dsh;
        sp += ph;
#pragma unroll
        for (int t = 0; t < V; ++t) {
          acc[t] = fmaf(dsh, kv[t], acc[t]);
          pk[t] = fmaf(ph, kv[t], pk[t]);
        }
      } else {
#pragma unroll
        for (int t = 0; t < V; ++t) acc[t] = fmaf(ds, kv[t], acc[t]);
      }
    }
  }
  if (!live) return;
  const float rho = GPROJ ? r / sp : 0.f;
#pragma unroll
  for (int t = 0; t < V; ++t) acc[t] = scale * (acc[t] - rho * pk[t]);
  store_vec(dQ + base + i * D, lane, acc);
  if (lane == 0) ws[tl.bh * N + i] = make_float4(Li, Di, rho, 0.f);
}

// ------------------------------------------------------- backward, columns
template <typename T, int D, bool GPROJ>
__global__ void __launch_bounds__(kThreads) bwd_col_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                           const T* __restrict__ Vt, const T* __restrict__ dO,
                                                           const float4* __restrict__ ws, T* __restrict__ dK,
                                                           T* __restrict__ dV, int64_t N, int64_t BHkv,
                                                           float scale, int causal, Band bd, int64_t G) {
  constexpr int V = D / 32;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Gs = sm + kTile * D;
  float4* Ss = reinterpret_cast<float4*>(sm + 2 * kTile * D);
  const int64_t nblk = (N + kWarps - 1) / kWarps;
  const Tile tl = decode(BHkv, nblk, false);  // tl.bh: a key/value head; smallest key index = most rows: first
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t col0 = tl.blk * kWarps, j = col0 + warp;
  // bd: the banded causal mask (key j is seen by the rows j <= i <= bd.key_hi(j))
  const int64_t hi_blk = causal ? bd.key_hi(tl.bh, lmin(col0 + kWarps - 1, N - 1)) : N - 1;  // last row any key sees
  const int64_t hi_j = causal ? bd.key_hi(tl.bh, j) : N - 1;
  const bool live = j < N;
  const size_t base = static_cast<size_t>(tl.bh) * N * D;
  float kv[V], vv[V], ak[V], av[V];
#pragma unroll
  for (int t = 0; t < V; ++t) ak[t] = av[t] = 0.f;
  if (live) {
    load_vec(K + base + j * D, lane, kv);
    load_vec(Vt + base + j * D, lane, vv);
  }
  // dK and dV of a shared head sum over the G query heads that read it.
  for (int64_t hq = tl.bh * G; hq < (tl.bh + 1) * G; ++hq)
  for (int64_t i0 = causal ? col0 : 0; i0 < (causal ? hi_blk + 1 : N); i0 += kTile) {
    const size_t qbase = static_cast<size_t>(hq) * N * D;
    __syncthreads();
    stage<T, D>(Qs, Q + qbase, i0, N);
    stage<T, D>(Gs, dO + qbase, i0, N);
    if (threadIdx.x < kTile)
      Ss[threadIdx.x] = (i0 + threadIdx.x < N) ? ws[hq * N + i0 + threadIdx.x] : make_float4(0, 0, 0, 0);
    __syncthreads();
    if (!live) continue;
    const int ib = causal ? static_cast<int>(lmax(0, j - i0)) : 0;  // causal: rows i >= j only
    const int ie = static_cast<int>(lmin(kTile, (causal ? hi_j + 1 : N) - i0));  // rows i <= bd.key_hi(j)
    for (int ii = ib; ii < ie; ++ii) {
      float qv[V], gv[V];
      load_smem(Qs + ii * D, lane, qv);
      load_smem(Gs + ii * D, lane, gv);
      const float4 st = Ss[ii];
      float x[2] = {dot(qv, kv), dot(gv, vv)};
      warp_sum(x);
      const float p = expf(x[0] * scale - st.x);
      const float ds = p * (x[1] - st.y);
      float cq, cv;
      if constexpr (GPROJ) {
        const float ph = bf16r(p);
        cq = bf16r(ds) - st.z * ph;
        cv = ph;
      } else {
        cq = ds;
        cv = p;
      }
#pragma unroll
      for (int t = 0; t < V; ++t) {
        ak[t] = fmaf(cq, qv[t], ak[t]);
        av[t] = fmaf(cv, gv[t], av[t]);
      }
    }
  }
  if (!live) return;
#pragma unroll
  for (int t = 0; t < V; ++t) ak[t] *= scale;
  store_vec(dK + base + j * D, lane, ak);
  store_vec(dV + base + j * D, lane, av);
}

// ------------------------------------------------------------- BoB, rows
// Streams keys past each query row; accumulates E, F' and X, Y, Z, U, and at the
// end applies the corrections that need the finished row:
//   gdO = X - E O,  gQ = s (Y - E Z - F' U),  F = F' - E D.
// GP (GProj, bf16): the dS of gQ's dS b product is rounded to bf16 as the tensor-core
// path rounds it and projected to zero row sum: Y gets bf16(dS) b, and rho_i (P^ b)_i is
// subtracted with rho_i = sum_j bf16(dS_ij) / sum_j bf16(P_ij); rho goes to rho_ws.
template <typename T, int D, bool GP>
__global__ void __launch_bounds__(kThreads) bob_row_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ Vt, const T* __restrict__ O,
    const T* __restrict__ dO, const float* __restrict__ lse, const T* __restrict__ A, const T* __restrict__ Bm,
    const T* __restrict__ C, T* __restrict__ gQ, T* __restrict__ gdO, float4* __restrict__ ws,
    float* __restrict__ rho_ws, int64_t N, int64_t BH, float scale, int causal, Band bd, int64_t G) {
  constexpr int V = D / 32;
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = sm + kTile * D;
  float* Bs = sm + 2 * kTile * D;
  float* Cs = sm + 3 * kTile * D;
  const int64_t nblk = (N + kWarps - 1) / kWarps;
  const Tile tl = decode(BH, nblk, true);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t row0 = tl.blk * kWarps, i = row0 + warp;
  const bool live = i < N;
  const size_t base = static_cast<size_t>(tl.bh) * N * D;
  const size_t kvbase = static_cast<size_t>(tl.bh / G) * N * D;  // K, V, b, c of the shared head
  float q[V], g[V], av[V], o[V], X[V], Y[V], Z[V], U[V], Pb[GP ? V : 1];
  float Di = 0.f, Li = 0.f, E = 0.f, Fp = 0.f, r = 0.f, sp = 0.f;
#pragma unroll
  for (int t = 0; t < V; ++t) X[t] = Y[t] = Z[t] = U[t] = 0.f;
#pragma unroll
  for (int t = 0; t < (GP ? V : 1); ++t) Pb[t] = 0.f;
  if (live) {
    load_vec(Q + base + i * D, lane, q);
    load_vec(dO + base + i * D, lane, g);
    load_vec(A + base + i * D, lane, av);
    load_vec(O + base + i * D, lane, o);
    float x[1] = {dot(g, o)};
    warp_sum(x);
    Di = x[0];
    Li = lse[tl.bh * N + i];
  }
  const int64_t last = causal ? min(row0 + kWarps, N) - 1 : N - 1;  // last key any row of the block sees
  // bd: the banded causal mask (row i sees the keys bd.row_lo(i) <= j <= i)
  const int64_t first = causal ? (bd.row_lo(tl.bh, row0) / kTile) * kTile : 0;  // first key tile any row sees
  const int64_t lo_i = causal ? bd.row_lo(tl.bh, i) : 0;  // this row's first visible key
  for (int64_t k0 = first; k0 <= last; k0 += kTile) {
    __syncthreads();
    stage<T, D>(Ks, K + kvbase, k0, N);
    stage<T, D>(Vs, Vt + kvbase, k0, N);
    stage<T, D>(Bs, Bm + kvbase, k0, N);
    stage<T, D>(Cs, C + kvbase, k0, N);
    __syncthreads();
    if (!live) continue;
    const int jn = static_cast<int>(lmin(kTile, (causal ? i + 1 : N) - k0));
    const int jb = causal ? static_cast<int>(lmin(kTile, lmax(0, lo_i - k0))) : 0;  // below the row's band
    for (int jj = jb; jj < jn; ++jj) {
      float kv[V], vv[V], bv[V], cv[V];
      load_smem(Ks + jj * D, lane, kv);
      load_smem(Vs + jj * D, lane, vv);
      load_smem(Bs + jj * D, lane, bv);
      load_smem(Cs + jj * D, lane, cv);
      float x[4] = {dot(q, kv), dot(g, vv), dot(av, kv) + dot(q, bv), dot(g, cv)};
      warp_sum(x);
      const float p = expf(x[0] * scale - Li);
      const float dp = x[1];
      const float G = scale * x[2];
      const float Hh = x[3];
      const float ds = p * (dp - Di);
      const float pg = p * G;
      const float w = G * ds + p * Hh;
      E += pg;
      Fp += w;
      const float dsb = GP ? bf16r(ds) : ds;  // the dS of the dS b product
      if constexpr (GP) {
        const float ph = bf16r(p);
        r += dsb;
        sp += ph;
#pragma unroll
        for (int t = 0; t < V; ++t) Pb[t] = fmaf(ph, bv[t], Pb[t]);
      }
#pragma unroll
      for (int t = 0; t < V; ++t) {
        X[t] = fmaf(p, cv[t], fmaf(pg, vv[t], X[t]));
        Y[t] = fmaf(dsb, bv[t], fmaf(w, kv[t], Y[t]));
        Z[t] = fmaf(ds, kv[t], Z[t]);
        U[t] = fmaf(p, kv[t], U[t]);
      }
    }
  }
  if (!live) return;
  const float rho = GP ? r / sp : 0.f;
  float go[V], gq[V];
#pragma unroll
  for (int t = 0; t < V; ++t) {
    go[t] = X[t] - E * o[t];
    gq[t] = scale * (Y[t] - E * Z[t] - Fp * U[t]);
    if constexpr (GP) gq[t] -= scale * rho * Pb[t];
  }
  store_vec(gdO + base + i * D, lane, go);
  store_vec(gQ + base + i * D, lane, gq);
  if (lane == 0) {
    ws[tl.bh * N + i] = make_float4(Li, Di, E, Fp - E * Di);
    if constexpr (GP) rho_ws[tl.bh * N + i] = rho;
  }
}

// ---------------------------------------------------------- BoB, columns
// GP: gK's dS^T a product sees the projected bf16(dS) - rho_i bf16(P) (rho from rho_ws).
template <typename T, int D, bool GP>
__global__ void __launch_bounds__(kThreads) bob_col_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ Vt, const T* __restrict__ dO,
    const T* __restrict__ A, const T* __restrict__ Bm, const T* __restrict__ C, const float4* __restrict__ ws,
    const float* __restrict__ rho_ws, T* __restrict__ gK, T* __restrict__ gV, int64_t N, int64_t BHkv,
    float scale, int causal, Band bd, int64_t G) {
  constexpr int V = D / 32;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Gs = sm + kTile * D;
  float* As = sm + 2 * kTile * D;
  float4* Ss = reinterpret_cast<float4*>(sm + 3 * kTile * D);
  float* Rs = reinterpret_cast<float*>(Ss + kTile);  // GP: rho of the staged rows
  const int64_t nblk = (N + kWarps - 1) / kWarps;
  const Tile tl = decode(BHkv, nblk, false);  // tl.bh: a key/value head
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t col0 = tl.blk * kWarps, j = col0 + warp;
  // bd: the banded causal mask (key j is seen by the rows j <= i <= bd.key_hi(j))
  const int64_t hi_blk = causal ? bd.key_hi(tl.bh, lmin(col0 + kWarps - 1, N - 1)) : N - 1;  // last row any key sees
  const int64_t hi_j = causal ? bd.key_hi(tl.bh, j) : N - 1;
  const bool live = j < N;
  const size_t base = static_cast<size_t>(tl.bh) * N * D;
  float kv[V], vv[V], bv[V], cv[V], aK[V], aV[V];
#pragma unroll
  for (int t = 0; t < V; ++t) aK[t] = aV[t] = 0.f;
  if (live) {
    load_vec(K + base + j * D, lane, kv);
    load_vec(Vt + base + j * D, lane, vv);
    load_vec(Bm + base + j * D, lane, bv);
    load_vec(C + base + j * D, lane, cv);
  }
  // gK and gV of a shared head sum over the G query heads that read it.
  for (int64_t hq = tl.bh * G; hq < (tl.bh + 1) * G; ++hq)
  for (int64_t i0 = causal ? col0 : 0; i0 < (causal ? hi_blk + 1 : N); i0 += kTile) {
    const size_t qbase = static_cast<size_t>(hq) * N * D;
    __syncthreads();
    stage<T, D>(Qs, Q + qbase, i0, N);
    stage<T, D>(Gs, dO + qbase, i0, N);
    stage<T, D>(As, A + qbase, i0, N);
    if (threadIdx.x < kTile) {
      Ss[threadIdx.x] = (i0 + threadIdx.x < N) ? ws[hq * N + i0 + threadIdx.x] : make_float4(0, 0, 0, 0);
      if constexpr (GP) Rs[threadIdx.x] = (i0 + threadIdx.x < N) ? rho_ws[hq * N + i0 + threadIdx.x] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    const int ib = causal ? static_cast<int>(lmax(0, j - i0)) : 0;
    const int ie = static_cast<int>(lmin(kTile, (causal ? hi_j + 1 : N) - i0));  // rows i <= bd.key_hi(j)
    for (int ii = ib; ii < ie; ++ii) {
      float qv[V], gv[V], a2[V];
      load_smem(Qs + ii * D, lane, qv);
      load_smem(Gs + ii * D, lane, gv);
      load_smem(As + ii * D, lane, a2);
      const float4 st = Ss[ii];  // (lse, D, E, F) of row i
      float x[4] = {dot(qv, kv), dot(gv, vv), dot(a2, kv) + dot(qv, bv), dot(gv, cv)};
      warp_sum(x);
      const float p = expf(x[0] * scale - st.x);
      const float dp = x[1];
      const float G = scale * x[2];
      const float Hh = x[3];
      const float ds = p * (dp - st.y);
      const float dpbar = p * (G - st.z);
      const float sbar = p * (G * (dp - st.y) - st.z * dp + Hh - st.w);
      const float dsa = GP ? bf16r(ds) - Rs[ii] * bf16r(p) : ds;  // the dS of the dS^T a product
#pragma unroll
      for (int t = 0; t < V; ++t) {
        aV[t] = fmaf(dpbar, gv[t], aV[t]);
        aK[t] = fmaf(dsa, a2[t], fmaf(sbar, qv[t], aK[t]));
      }
    }
  }
  if (!live) return;
#pragma unroll
  for (int t = 0; t < V; ++t) aK[t] *= scale;
  store_vec(gK + base + j * D, lane, aK);
  store_vec(gV + base + j * D, lane, aV);
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

template <typename Kern>
cudaError_t allow_smem(Kern k, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

inline unsigned grid_for(const Problem& p) {
  return static_cast<unsigned>(((p.N + kWarps - 1) / kWarps) * p.BH);
}
// Column passes: one CTA per block of keys of one key/value head.
inline unsigned grid_for_cols(const Problem& p) {
  return static_cast<unsigned>(((p.N + kWarps - 1) / kWarps) * p.BHkv);
}

template <typename T, int D, bool GP>
cudaError_t bwd_t(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes, cudaStream_t st) {
  const size_t sm_row = 2 * kTile * D * sizeof(float);
  const size_t sm_col = 2 * kTile * D * sizeof(float) + kTile * sizeof(float4);
  auto kr = bwd_row_kernel<T, D, GP>;
  auto kc = bwd_col_kernel<T, D, GP>;
  cudaError_t e = allow_smem(kr, sm_row);
  if (e == cudaSuccess) e = allow_smem(kc, sm_col);
  if (e != cudaSuccess) return e;
  if (passes & 1) {
    kr<<<grid_for(p), kThreads, sm_row, st>>>(static_cast<const T*>(Q), static_cast<const T*>(K),
                                               static_cast<const T*>(V), static_cast<const T*>(O),
                                               static_cast<const T*>(dO), lse, static_cast<T*>(dQ), ws, p.N, p.BH,
                                               p.scale, p.causal, make_band(p, eff_window(p), false), p.group);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!(passes & 2)) return cudaSuccess;
  kc<<<grid_for_cols(p), kThreads, sm_col, st>>>(static_cast<const T*>(Q), static_cast<const T*>(K),
                                                  static_cast<const T*>(V), static_cast<const T*>(dO), ws,
                                                  static_cast<T*>(dK), static_cast<T*>(dV), p.N, p.BHkv, p.scale,
                                                  p.causal, make_band(p, eff_window(p), true), p.group);
  return cudaGetLastError();
}

template <typename T, int D, bool GP>
cudaError_t bob_t(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* lse, const void* a, const void* b, const void* c, void* gQ, void* gK, void* gV,
                  void* gdO, float4* ws, float* rho_ws, int passes, cudaStream_t st) {
  const size_t sm_row = 4 * kTile * D * sizeof(float);
  const size_t sm_col = 3 * kTile * D * sizeof(float) + kTile * (sizeof(float4) + sizeof(float));
  auto kr = bob_row_kernel<T, D, GP>;
  auto kc = bob_col_kernel<T, D, GP>;
  cudaError_t e = allow_smem(kr, sm_row);
  if (e == cudaSuccess) e = allow_smem(kc, sm_col);
  if (e != cudaSuccess) return e;
  using CT = const T*;
  if (passes & 1) {
    kr<<<grid_for(p), kThreads, sm_row, st>>>(
        static_cast<CT>(Q), static_cast<CT>(K), static_cast<CT>(V), static_cast<CT>(O), static_cast<CT>(dO), lse,
        static_cast<CT>(a), static_cast<CT>(b), static_cast<CT>(c), static_cast<T*>(gQ), static_cast<T*>(gdO), ws,
        rho_ws, p.N, p.BH, p.scale, p.causal, make_band(p, eff_window(p), false), p.group);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!(passes & 2)) return cudaSuccess;
  kc<<<grid_for_cols(p), kThreads, sm_col, st>>>(static_cast<CT>(Q), static_cast<CT>(K), static_cast<CT>(V),
                                                  static_cast<CT>(dO), static_cast<CT>(a), static_cast<CT>(b),
                                                  static_cast<CT>(c), ws, rho_ws, static_cast<T*>(gK),
                                                  static_cast<T*>(gV), p.N, p.BHkv, p.scale, p.causal, make_band(p, eff_window(p), true), p.group);
  return cudaGetLastError();
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

// Element type of the [B,H,N,d] tensors this path serves: bf16 (float32 inputs have
// tensor-core kernels at every head dim; for them the launchers return an error).
template <typename F>
void with_type(int dtype, F&& f) {
  if (dtype == ATTN_BF16) f(__nv_bfloat16{});
}

cudaError_t simt_bwd(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                     const void* dO, const float* lse, void* dQ, void* dK, void* dV, int gproj, float4* ws,
                     int passes, cudaStream_t st) {
  // float32 dS is never rounded, so GProj applies to bf16 only (its rounding is emulated).
  const bool gp = gproj != 0 && p.dtype == ATTN_BF16;
  cudaError_t e = cudaErrorInvalidValue;
  with_type(p.dtype, [&](auto t) {
    using T = decltype(t);
    with_head_dim(p.d, [&](auto dd) {
      e = gp ? bwd_t<T, dd(), true>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st)
             : bwd_t<T, dd(), false>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st);
    });
  });
  return e;
}

cudaError_t simt_bob(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                     const void* dO, const float* lse, const void* a, const void* b, const void* c, void* gQ,
                     void* gK, void* gV, void* gdO, bool gproj, float4* ws, int passes, cudaStream_t st) {
  // GProj applies to bf16 only (float32 dS is never rounded); its coefficients follow the
  // row states in the workspace (internal.h; this path keeps one float per row there).
  float* rho_ws = reinterpret_cast<float*>(bob_rho_region(ws, p));
  cudaError_t e = cudaErrorInvalidValue;
  with_type(p.dtype, [&](auto t) {
    using T = decltype(t);
    with_head_dim(p.d, [&](auto dd) {
      if constexpr (std::is_same_v<T, __nv_bfloat16>) {
        if (gproj) {
          e = bob_t<T, dd(), true>(p, Q, K, V, O, dO, lse, a, b, c, gQ, gK, gV, gdO, ws, rho_ws, passes, st);
          return;
        }
      }
      e = bob_t<T, dd(), false>(p, Q, K, V, O, dO, lse, a, b, c, gQ, gK, gV, gdO, ws, nullptr, passes, st);
    });
  });
  return e;
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
