// float32 attention on the tcgen05 tensor cores (kind::tf32), d = 32 and 64: forward,
// backward (row and column passes) and BoB (row and column passes), the same
// decomposition as the bf16 kernels and the CUDA-core float32 kernels:
//   forward   online softmax ("Flash attention for trading models", "Online softmax
//             recurrence"), O and the natural-log lse written once;
//   backward  P recomputed from lse ("Backward pass: recompute instead of store"):
//             row pass dQ = s dS K with dS = P (dP - D), D_i = dO_i . O_i; column
//             pass dV = P^T dO, dK = s dS^T Q;
//   BoB       ("FlashBoB: second-order attention", "Two scalar states replace
//             quadratic tensors"): the row pass accumulates X = P c + (P G) V,
//             Y = W K + dS b, Z = dS K, U = P K and the states E = sum P G,
//             F' = sum W, and writes gdO = X - E O, gQ = s (Y - E Z - F' U); the
//             column pass re-reads (lse, D, E, F = F' - E D) and accumulates
//             gV = dPbar^T dO, gK = s (dS^T a + Sbar^T Q), with G = s (a K^T + Q b^T),
//             H = dO c^T, W = G dS + P H, dPbar = P (G - E),
//             Sbar = P (G (dP - D) - E dP + H - F).
//
// Precision: every product A B^T runs as three tf32 products,
//   A B^T ~ A_lo B_hi^T + A_hi B_lo^T + A_hi B_hi^T,
// with x_hi = tf32(x) and x_lo = tf32(x - x_hi) (round to nearest), so each element
// product is exact to about 2^-21 relative (the dropped A_lo B_lo term and the rounding
// of the low parts), accumulated in fp32 in tensor memory.  Everything else (softmax,
// the elementwise terms, the states) is fp32 on the CUDA cores with expf.
//
// Structure: one CTA of 128 threads holds 128 rows (queries in row passes, keys in
// column passes), one row per thread and per TMEM lane, and streams blocks of 64
// partner rows.  Each product is one synchronous step: the threads write the two
// operands into 128-byte-swizzled K-major shared-memory tiles (A: 128 rows, B: 64 or d
// rows, K up to 64 fp32 in two 128-byte slabs), split into their tf32 high and low
// parts; one warp issues the MMAs and commits them to an mbarrier that every thread
// waits on (bounded).  Operands that are products of the threads' own rows (P, dS, ...)
// are written from registers or copied back from TMEM into the A tile; the transposed
// streamed operands (V^T, K^T, dO^T, ...) are transposed while they are split.  The
// float32 path is the precision path (its tolerance is 1e-5, not its speed), so the
// steps are not overlapped.
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fbd {
namespace {

__device__ unsigned int g_err = 0;

constexpr int BM = 128;  // rows held per CTA: one per thread and per TMEM lane
constexpr int BN = 64;   // rows of a streamed block
constexpr int kThreads = 128;
constexpr int kA = BM * 64 * 4;  // A tile, one part: 128 rows x 64 fp32
constexpr int kB = BN * 64 * 4;  // B tile, one part: 64 rows x 64 fp32
constexpr int oAh = 0, oAl = kA, oBh = 2 * kA, oBl = 2 * kA + kB;
constexpr int oSt = 2 * kA + 2 * kB;  // 64 row states (float4) of the streamed block
constexpr int oBar = oSt + BN * 16;
constexpr int kSmem = oBar + 64;
// The BoB passes take all 512 TMEM columns: their CTAs ask for more shared memory than
// two CTAs could share, so that no second CTA on the SM waits for columns.
constexpr int kSmemBob = 120 * 1024;
static_assert(kSmem <= kSmemBob && kSmemBob <= 232448, "shared memory");

using tc::f;

struct Ctx {
  uint8_t* sm;
  uint32_t tmem;
  uint64_t* bar;
  volatile int* abort_flag;
  uint32_t phase;
};

__device__ __forceinline__ Ctx setup(uint8_t* sm, uint32_t ncols) {
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + oBar);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    // The swizzled operand layout needs 1024-byte aligned tiles.
    *abort_flag = (ptx::smem_u32(sm) & 1023u) ? 1 : 0;
    if (*abort_flag) atomicOr(&g_err, FBD_ERR_TIMEOUT);
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    ptx::tmem_alloc(slot, ncols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return Ctx{sm, *slot, bar, abort_flag, 0};
}

__device__ __forceinline__ void teardown(const Ctx& c, uint32_t ncols) {
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(c.tmem, ncols);
  }
}

// Byte offset of element (row, k) in a K-major tile of R rows: k in slabs of 32 fp32
// (128 bytes per row), 16-byte chunks swizzled by the row within its 8-row group.
__device__ __forceinline__ int swz(int row, int k, int R) {
  return (k >> 5) * R * 128 + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) + ((k & 3) << 2);
}

// Four consecutive K elements of one row, split into tf32 high and low parts.
__device__ __forceinline__ void put4(uint8_t* hi, uint8_t* lo, int off, float4 v) {
  const float4 h = make_float4(ptx::to_tf32(v.x), ptx::to_tf32(v.y), ptx::to_tf32(v.z), ptx::to_tf32(v.w));
  const float4 l = make_float4(ptx::to_tf32(v.x - h.x), ptx::to_tf32(v.y - h.y), ptx::to_tf32(v.z - h.z),
                               ptx::to_tf32(v.w - h.w));
  *reinterpret_cast<float4*>(hi + off) = h;
  *reinterpret_cast<float4*>(lo + off) = l;
}
__device__ __forceinline__ void put1(uint8_t* hi, uint8_t* lo, int off, float v) {
  const float h = ptx::to_tf32(v);
  *reinterpret_cast<float*>(hi + off) = h;
  *reinterpret_cast<float*>(lo + off) = ptx::to_tf32(v - h);
}

// R rows (row0 ...) of a row-major [rows][KD] fp32 array as a K-major tile (K = KD);
// rows at or past `nrows` are zero.  `a`: the A tile (else the B tile).
template <int KD>
__device__ __forceinline__ void stage_rows(const Ctx& c, bool a, const float* src, int64_t row0, int64_t nrows,
                                           int R) {
  constexpr int C4 = KD / 4;
  uint8_t* hi = c.sm + (a ? oAh : oBh);
  uint8_t* lo = c.sm + (a ? oAl : oBl);
  for (int idx = threadIdx.x; idx < R * C4; idx += kThreads) {
    const int row = idx / C4, k = (idx % C4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + row < nrows) v = *reinterpret_cast<const float4*>(src + (row0 + row) * KD + k);
    put4(hi, lo, swz(row, k, R), v);
  }
}

// 64 rows (row0 ...) of a row-major [rows][KD] array, transposed: the B tile of KD rows
// whose K index is the source row (for the products with K = the streamed rows).
template <int KD>
__device__ __forceinline__ void stage_rows_t(const Ctx& c, const float* src, int64_t row0, int64_t nrows) {
  constexpr int C4 = KD / 4;
  uint8_t* hi = c.sm + oBh;
  uint8_t* lo = c.sm + oBl;
  for (int idx = threadIdx.x; idx < BN * C4; idx += kThreads) {
    const int srow = idx / C4, col = (idx % C4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + srow < nrows) v = *reinterpret_cast<const float4*>(src + (row0 + srow) * KD + col);
    put1(hi, lo, swz(col, srow, KD), v.x);
    put1(hi, lo, swz(col + 1, srow, KD), v.y);
    put1(hi, lo, swz(col + 2, srow, KD), v.z);
    put1(hi, lo, swz(col + 3, srow, KD), v.w);
  }
}

// Row threadIdx.x of the A tile (K = 64) from 32 values at K offset k0.
__device__ __forceinline__ void stage_own(const Ctx& c, int k0, const float (&v)[32]) {
  const int r = threadIdx.x;
#pragma unroll
  for (int k = 0; k < 32; k += 4)
    put4(c.sm + oAh, c.sm + oAl, swz(r, k0 + k, BM), make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]));
}

__device__ __forceinline__ uint32_t lane_base() { return static_cast<uint32_t>(threadIdx.x & ~31) << 16; }

// 32 fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tld(const Ctx& c, uint32_t col, float (&v)[32]) {
  uint32_t u[32];
  ptx::tmem_ld32(c.tmem + lane_base() + col, u);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int t = 0; t < 32; ++t) v[t] = f(u[t]);
}
__device__ __forceinline__ void tst(const Ctx& c, uint32_t col, const float (&v)[32]) {
  uint32_t u[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) u[t] = __float_as_uint(v[t]);
  ptx::tmem_st32(c.tmem + lane_base() + col, u);
  ptx::tmem_wait_st();
}

// The A tile (K = 64) from 64 TMEM columns of this thread's lane.
__device__ __forceinline__ void stage_tmem(const Ctx& c, uint32_t col) {
  float v[32];
  tld(c, col, v);
  stage_own(c, 0, v);
  tld(c, col + 32, v);
  stage_own(c, 32, v);
}

// TMEM columns [col, col + n) (+)= A B^T over nk K-steps of 8: A = the A tile (128
// rows), B = the B tile (n rows).  Synchronous: returns when the products are done.
__device__ __forceinline__ void mma3(Ctx& c, uint32_t col, int n, int nk, bool accumulate) {
  ptx::fence_proxy_async_smem();  // the threads' shared-memory writes, visible to the MMA
  ptx::tc_fence_before();         // and their TMEM reads and writes ordered before it
  __syncthreads();
  if (threadIdx.x < 32 && *c.abort_flag == 0) {
    ptx::tc_fence_after();
    const uint32_t id = ptx::idesc_tf32(BM, n);
    const uint32_t ah = ptx::smem_u32(c.sm + oAh), al = ptx::smem_u32(c.sm + oAl);
    const uint32_t bh = ptx::smem_u32(c.sm + oBh), bl = ptx::smem_u32(c.sm + oBl);
    for (int k = 0; k < nk; ++k) {
      const uint64_t dah = tc::kmajor_desc(ah, BM, k), dal = tc::kmajor_desc(al, BM, k);
      const uint64_t dbh = tc::kmajor_desc(bh, n, k), dbl = tc::kmajor_desc(bl, n, k);
      ptx::mma_ss_tf32_e(c.tmem + col, dal, dbh, id, (accumulate || k > 0) ? 1u : 0u);
      ptx::mma_ss_tf32_e(c.tmem + col, dah, dbl, id, 1u);
      ptx::mma_ss_tf32_e(c.tmem + col, dah, dbh, id, 1u);
    }
    ptx::mma_commit_e(c.bar);
  }
  const ptx::BoundedWait wait{c.abort_flag, &g_err};
  wait(c.bar, c.phase & 1);
  ++c.phase;
  ptx::tc_fence_after();
}

// Running accumulator (TMEM columns acc .. acc + D) += the block product in the scratch
// columns, in IEEE fp32 on the CUDA cores (first: the accumulator takes the product).
// The tensor core's own accumulation rounds differently from fp32 addition, and its
// error grows with the length of the chain; across blocks the sums are kept here.
template <int D>
__device__ __forceinline__ void add_into(const Ctx& c, uint32_t acc, uint32_t scr, bool first) {
#pragma unroll 1
  for (int h = 0; h < D / 32; ++h) {
    float t[32];
    tld(c, scr + 32 * h, t);
    if (!first) {
      float a[32];
      tld(c, acc + 32 * h, a);
#pragma unroll
      for (int u = 0; u < 32; ++u) t[u] += a[u];
    }
    tst(c, acc + 32 * h, t);
  }
}
// One block's output product into the scratch columns, then into the accumulator.
template <int D>
__device__ __forceinline__ void mma_acc(Ctx& c, uint32_t acc, uint32_t scr, bool first) {
  mma3(c, scr, D, BN / 8, false);
  add_into<D>(c, acc, scr, first);
}

template <int D>
__device__ __forceinline__ void load_row(const float* src, float (&v)[D]) {
#pragma unroll
  for (int k = 0; k < D; k += 4) {
    const float4 x = *reinterpret_cast<const float4*>(src + k);
    v[k] = x.x;
    v[k + 1] = x.y;
    v[k + 2] = x.z;
    v[k + 3] = x.w;
  }
}
template <int D>
__device__ __forceinline__ void store_row(float* dst, const float (&v)[D]) {
#pragma unroll
  for (int k = 0; k < D; k += 4) *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
}
// D accumulator columns of this thread's lane (D = 32 or 64), times `mul`.
template <int D>
__device__ __forceinline__ void tld_acc(const Ctx& c, uint32_t col, float mul, float (&v)[D]) {
  float t[32];
#pragma unroll
  for (int h = 0; h < D / 32; ++h) {
    tld(c, col + 32 * h, t);
#pragma unroll
    for (int u = 0; u < 32; ++u) v[32 * h + u] = mul * t[u];
  }
}

// Key blocks of a row block (row passes) and query blocks of a key block (column
// passes) under the mask; bd gives each row's first key and each key's last row.
struct RowRange {
  int k0, k1;
};
__device__ __forceinline__ RowRange key_blocks(int rb, int N, int causal, const Band& bd, int bh) {
  if (!causal) return {0, (N + BN - 1) / BN};
  return {bd.row_lo(bh, static_cast<int64_t>(rb) * BM) / BN, min(rb * BM + BM - 1, N - 1) / BN + 1};
}
__device__ __forceinline__ RowRange query_blocks(int kb, int N, int causal, const Band& bd, int kvh) {
  if (!causal) return {0, (N + BN - 1) / BN};
  return {kb * BM / BN, bd.key_hi(kvh, min(kb * BM + BM - 1, N - 1)) / BN + 1};
}

// ------------------------------------------------------------------ forward
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_fwd_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
                   float* __restrict__ O, float* __restrict__ lse, int N, int nrb, int BH, float scale, int causal,
                   Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  Ctx c = setup(sm, 128);  // S / P 0-63, P V 64-127
  const tc::Order ord = tc::grid_order(BH, nrb);
  const int bh = ord.bh, rb = nrb - 1 - ord.k, kvh = bh / G;
  const int64_t i = static_cast<int64_t>(rb) * BM + threadIdx.x;
  const float* q = Q + static_cast<size_t>(bh) * N * D;
  const float* k = K + static_cast<size_t>(kvh) * N * D;
  const float* v = V + static_cast<size_t>(kvh) * N * D;
  const int lo_i = causal ? bd.row_lo(bh, i) : 0;
  const RowRange rr = key_blocks(rb, N, causal, bd, bh);
  float m = -INFINITY, l = 0.f, o[D];
#pragma unroll
  for (int t = 0; t < D; ++t) o[t] = 0.f;
  for (int kb = rr.k0; kb < rr.k1; ++kb) {
    stage_rows<D>(c, true, q, static_cast<int64_t>(rb) * BM, N, BM);
    stage_rows<D>(c, false, k, static_cast<int64_t>(kb) * BN, N, BN);
    mma3(c, 0, BN, D / 8, false);  // S = Q K^T
    float s[2][32];
    tld(c, 0, s[0]);
    tld(c, 32, s[1]);
    float mx = -INFINITY;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int64_t key = static_cast<int64_t>(kb) * BN + 32 * h + t;
        const bool vis = i < N && key < N && (!causal || (key <= i && key >= lo_i));
        s[h][t] = vis ? s[h][t] * scale : -INFINITY;
        mx = fmaxf(mx, s[h][t]);
      }
    const float m_new = fmaxf(m, mx);
    // No visible key yet (the row's band starts later): p = 0, nothing rescaled.
    const float alpha = m_new == -INFINITY ? 1.f : expf(m - m_new);
    float rs = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        s[h][t] = s[h][t] == -INFINITY ? 0.f : expf(s[h][t] - m_new);
        rs += s[h][t];
      }
      stage_own(c, 32 * h, s[h]);
    }
    m = m_new;
    l = l * alpha + rs;
    stage_rows_t<D>(c, v, static_cast<int64_t>(kb) * BN, N);
    mma3(c, 64, D, BN / 8, false);  // P V
#pragma unroll
    for (int h = 0; h < D / 32; ++h) {
      float pv[32];
      tld(c, 64 + 32 * h, pv);
#pragma unroll
      for (int t = 0; t < 32; ++t) o[32 * h + t] = o[32 * h + t] * alpha + pv[t];
    }
  }
  if (i < N) {
    const float inv = 1.f / l;
#pragma unroll
    for (int t = 0; t < D; ++t) o[t] *= inv;
    store_row<D>(O + (static_cast<size_t>(bh) * N + i) * D, o);
    lse[static_cast<size_t>(bh) * N + i] = m + logf(l);
  }
  teardown(c, 128);
}

// --------------------------------------------------------- backward, rows
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bwd_row_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
                       const float* __restrict__ O, const float* __restrict__ dO, const float* __restrict__ lse,
                       float* __restrict__ dQ, float4* __restrict__ ws, int N, int nrb, int BH, float scale,
                       int causal, Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  Ctx c = setup(sm, 256);  // S 0-63, dP 64-127, dQ 128-191
  const tc::Order ord = tc::grid_order(BH, nrb);
  const int bh = ord.bh, rb = nrb - 1 - ord.k, kvh = bh / G;
  const int64_t i = static_cast<int64_t>(rb) * BM + threadIdx.x;
  const size_t qo = static_cast<size_t>(bh) * N * D, ko = static_cast<size_t>(kvh) * N * D;
  const int lo_i = causal ? bd.row_lo(bh, i) : 0;
  float Di = 0.f, Li = 0.f;
  if (i < N) {
    float a[D], b[D];
    load_row<D>(dO + qo + i * D, a);
    load_row<D>(O + qo + i * D, b);
#pragma unroll
    for (int t = 0; t < D; ++t) Di = fmaf(a[t], b[t], Di);
    Li = lse[static_cast<size_t>(bh) * N + i];
  }
  const RowRange rr = key_blocks(rb, N, causal, bd, bh);
  for (int kb = rr.k0; kb < rr.k1; ++kb) {
    const int64_t k0 = static_cast<int64_t>(kb) * BN;
    stage_rows<D>(c, true, Q + qo, static_cast<int64_t>(rb) * BM, N, BM);
    stage_rows<D>(c, false, K + ko, k0, N, BN);
    mma3(c, 0, BN, D / 8, false);  // S = Q K^T
    stage_rows<D>(c, true, dO + qo, static_cast<int64_t>(rb) * BM, N, BM);
    stage_rows<D>(c, false, V + ko, k0, N, BN);
    mma3(c, 64, BN, D / 8, false);  // dP = dO V^T
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float s[32], dp[32];
      tld(c, 32 * h, s);
      tld(c, 64 + 32 * h, dp);
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int64_t key = k0 + 32 * h + t;
        const bool vis = i < N && key < N && (!causal || (key <= i && key >= lo_i));
        s[t] = vis ? expf(s[t] * scale - Li) * (dp[t] - Di) : 0.f;  // dS
      }
      stage_own(c, 32 * h, s);
    }
    stage_rows_t<D>(c, K + ko, k0, N);
    mma_acc<D>(c, 128, 0, kb == rr.k0);  // dQ += dS K (S and dP are read: scratch at 0)
  }
  float g[D];
  tld_acc<D>(c, 128, scale, g);
  if (i < N) {
    store_row<D>(dQ + qo + i * D, g);
    ws[static_cast<size_t>(bh) * N + i] = make_float4(Li, Di, 0.f, 0.f);
  }
  teardown(c, 256);
}

// ------------------------------------------------------- backward, columns
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bwd_col_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
                       const float* __restrict__ dO, const float4* __restrict__ ws, float* __restrict__ dK,
                       float* __restrict__ dV, int N, int nkb, int BHkv, float scale, int causal, Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  Ctx c = setup(sm, 256);  // S^T / P^T 0-63, dP^T / dS^T 64-127, dV 128-191, dK 192-255
  const tc::Order ord = tc::grid_order(BHkv, nkb);
  const int kvh = ord.bh, kb = ord.k;
  const int64_t key = static_cast<int64_t>(kb) * BM + threadIdx.x;
  const size_t ko = static_cast<size_t>(kvh) * N * D;
  const int hi_k = causal ? bd.key_hi(kvh, key) : N - 1;
  const RowRange qr = query_blocks(kb, N, causal, bd, kvh);
  const float4* st = reinterpret_cast<const float4*>(sm + oSt);
  bool first = true;
  for (int hq = kvh * G; hq < (kvh + 1) * G; ++hq) {
    const size_t qo = static_cast<size_t>(hq) * N * D;
    for (int qb = qr.k0; qb < qr.k1; ++qb) {
      const int64_t q0 = static_cast<int64_t>(qb) * BN;
      if (threadIdx.x < BN) {
        const int64_t qi = q0 + threadIdx.x;
        reinterpret_cast<float4*>(sm + oSt)[threadIdx.x] =
            qi < N ? ws[static_cast<size_t>(hq) * N + qi] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      stage_rows<D>(c, true, K + ko, static_cast<int64_t>(kb) * BM, N, BM);
      stage_rows<D>(c, false, Q + qo, q0, N, BN);
      mma3(c, 0, BN, D / 8, false);  // S^T = K Q^T (the barrier in mma3 also publishes the states)
      stage_rows<D>(c, true, V + ko, static_cast<int64_t>(kb) * BM, N, BM);
      stage_rows<D>(c, false, dO + qo, q0, N, BN);
      mma3(c, 64, BN, D / 8, false);  // dP^T = V dO^T
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float s[32], dp[32];
        tld(c, 32 * h, s);
        tld(c, 64 + 32 * h, dp);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int64_t qi = q0 + 32 * h + t;
          const float4 sv = st[32 * h + t];  // (lse, D) of query qi
          const bool vis = key < N && qi < N && (!causal || (qi >= key && qi <= hi_k));
          const float p = vis ? expf(s[t] * scale - sv.x) : 0.f;
          s[t] = p;
          dp[t] = p * (dp[t] - sv.y);  // dS
        }
        stage_own(c, 32 * h, s);  // P^T
        tst(c, 64 + 32 * h, dp);
      }
      stage_rows_t<D>(c, dO + qo, q0, N);
      mma_acc<D>(c, 128, 0, first);  // dV += P^T dO (P^T is in the A tile: scratch at 0)
      stage_tmem(c, 64);
      stage_rows_t<D>(c, Q + qo, q0, N);
      mma_acc<D>(c, 192, 0, first);  // dK += dS^T Q
      first = false;
    }
  }
  float gv[D], gk[D];
  tld_acc<D>(c, 128, 1.f, gv);
  tld_acc<D>(c, 192, scale, gk);
  if (key < N) {
    store_row<D>(dV + ko + key * D, gv);
    store_row<D>(dK + ko + key * D, gk);
  }
  teardown(c, 256);
}

// ------------------------------------------------------------------ BoB, rows
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bob_row_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
                       const float* __restrict__ O, const float* __restrict__ dO, const float* __restrict__ lse,
                       const float* __restrict__ A, const float* __restrict__ Bm, const float* __restrict__ C,
                       float* __restrict__ gQ, float* __restrict__ gdO, float4* __restrict__ ws, int N, int nrb,
                       int BH, float scale, int causal, Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  // TMEM: S / P 0, dP / dS 64, G / PG 128, H / W 192, X 256, Y 320, Z 384, U 448.
  Ctx c = setup(sm, 512);
  const tc::Order ord = tc::grid_order(BH, nrb);
  const int bh = ord.bh, rb = nrb - 1 - ord.k, kvh = bh / G;
  const int64_t i = static_cast<int64_t>(rb) * BM + threadIdx.x;
  const int64_t r0 = static_cast<int64_t>(rb) * BM;
  const size_t qo = static_cast<size_t>(bh) * N * D, ko = static_cast<size_t>(kvh) * N * D;
  const int lo_i = causal ? bd.row_lo(bh, i) : 0;
  float Di = 0.f, Li = 0.f, E = 0.f, Fp = 0.f;
  if (i < N) {
    float a[D], b[D];
    load_row<D>(dO + qo + i * D, a);
    load_row<D>(O + qo + i * D, b);
#pragma unroll
    for (int t = 0; t < D; ++t) Di = fmaf(a[t], b[t], Di);
    Li = lse[static_cast<size_t>(bh) * N + i];
  }
  const RowRange rr = key_blocks(rb, N, causal, bd, bh);
  for (int kb = rr.k0; kb < rr.k1; ++kb) {
    const int64_t k0 = static_cast<int64_t>(kb) * BN;
    const bool acc = kb > rr.k0;
    stage_rows<D>(c, true, Q + qo, r0, N, BM);
    stage_rows<D>(c, false, K + ko, k0, N, BN);
    mma3(c, 0, BN, D / 8, false);  // S = Q K^T
    stage_rows<D>(c, false, Bm + ko, k0, N, BN);
    mma3(c, 128, BN, D / 8, false);  // G = Q b^T ...
    stage_rows<D>(c, true, A + qo, r0, N, BM);
    stage_rows<D>(c, false, K + ko, k0, N, BN);
    mma3(c, 128, BN, D / 8, true);  // ... + a K^T
    stage_rows<D>(c, true, dO + qo, r0, N, BM);
    stage_rows<D>(c, false, V + ko, k0, N, BN);
    mma3(c, 64, BN, D / 8, false);  // dP = dO V^T
    stage_rows<D>(c, false, C + ko, k0, N, BN);
    mma3(c, 192, BN, D / 8, false);  // H = dO c^T
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float s[32], dp[32], g[32], hh[32];
      tld(c, 32 * h, s);
      tld(c, 64 + 32 * h, dp);
      tld(c, 128 + 32 * h, g);
      tld(c, 192 + 32 * h, hh);
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int64_t key = k0 + 32 * h + t;
        const bool vis = i < N && key < N && (!causal || (key <= i && key >= lo_i));
        const float p = vis ? expf(s[t] * scale - Li) : 0.f;
        const float gg = scale * g[t];
        const float ds = p * (dp[t] - Di);
        const float pg = p * gg;
        const float w = gg * ds + p * hh[t];
        E += pg;
        Fp += w;
        s[t] = p;
        dp[t] = ds;
        g[t] = pg;
        hh[t] = w;
      }
      tst(c, 32 * h, s);
      tst(c, 64 + 32 * h, dp);
      tst(c, 128 + 32 * h, g);
      tst(c, 192 + 32 * h, hh);
    }
    // Block products into the scratch columns 0-63 (P, once in the A tile, is not read
    // from TMEM again), each added to its accumulator.
    stage_tmem(c, 0);  // P
    stage_rows_t<D>(c, C + ko, k0, N);
    mma_acc<D>(c, 256, 0, !acc);  // X += P c
    stage_rows_t<D>(c, K + ko, k0, N);
    mma_acc<D>(c, 448, 0, !acc);  // U += P K
    stage_tmem(c, 128);  // P G
    stage_rows_t<D>(c, V + ko, k0, N);
    mma_acc<D>(c, 256, 0, false);  // X += (P G) V
    stage_tmem(c, 64);  // dS
    stage_rows_t<D>(c, K + ko, k0, N);
    mma_acc<D>(c, 384, 0, !acc);  // Z += dS K
    stage_rows_t<D>(c, Bm + ko, k0, N);
    mma_acc<D>(c, 320, 0, !acc);  // Y += dS b
    stage_tmem(c, 192);  // W
    stage_rows_t<D>(c, K + ko, k0, N);
    mma_acc<D>(c, 320, 0, false);  // Y += W K
  }
#pragma unroll 1
  for (int h = 0; h < D / 32; ++h) {  // 32 output columns at a time
    float x[32], y[32], z[32], u[32];
    tld(c, 256 + 32 * h, x);
    tld(c, 320 + 32 * h, y);
    tld(c, 384 + 32 * h, z);
    tld(c, 448 + 32 * h, u);
    if (i < N) {
      float o[32];
      load_row<32>(O + qo + i * D + 32 * h, o);
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        x[t] = x[t] - E * o[t];                        // gdO
        y[t] = scale * (y[t] - E * z[t] - Fp * u[t]);  // gQ
      }
      store_row<32>(gdO + qo + i * D + 32 * h, x);
      store_row<32>(gQ + qo + i * D + 32 * h, y);
    }
  }
  if (i < N) ws[static_cast<size_t>(bh) * N + i] = make_float4(Li, Di, E, Fp - E * Di);
  teardown(c, 512);
}

// --------------------------------------------------------------- BoB, columns
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bob_col_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
                       const float* __restrict__ dO, const float* __restrict__ A, const float* __restrict__ Bm,
                       const float* __restrict__ C, const float4* __restrict__ ws, float* __restrict__ gK,
                       float* __restrict__ gV, int N, int nkb, int BHkv, float scale, int causal, Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  // TMEM: S^T / dPbar 0, dP^T / dS 64, G^T / Sbar 128, H^T 192, gV 256, gK 320, scratch 384.
  Ctx c = setup(sm, 512);
  const tc::Order ord = tc::grid_order(BHkv, nkb);
  const int kvh = ord.bh, kb = ord.k;
  const int64_t key = static_cast<int64_t>(kb) * BM + threadIdx.x;
  const int64_t c0 = static_cast<int64_t>(kb) * BM;
  const size_t ko = static_cast<size_t>(kvh) * N * D;
  const int hi_k = causal ? bd.key_hi(kvh, key) : N - 1;
  const RowRange qr = query_blocks(kb, N, causal, bd, kvh);
  const float4* st = reinterpret_cast<const float4*>(sm + oSt);
  bool first = true;
  for (int hq = kvh * G; hq < (kvh + 1) * G; ++hq) {
    const size_t qo = static_cast<size_t>(hq) * N * D;
    for (int qb = qr.k0; qb < qr.k1; ++qb) {
      const int64_t q0 = static_cast<int64_t>(qb) * BN;
      if (threadIdx.x < BN) {
        const int64_t qi = q0 + threadIdx.x;
        reinterpret_cast<float4*>(sm + oSt)[threadIdx.x] =
            qi < N ? ws[static_cast<size_t>(hq) * N + qi] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      stage_rows<D>(c, true, K + ko, c0, N, BM);
      stage_rows<D>(c, false, Q + qo, q0, N, BN);
      mma3(c, 0, BN, D / 8, false);  // S^T = K Q^T (the barrier in mma3 also publishes the states)
      stage_rows<D>(c, false, A + qo, q0, N, BN);
      mma3(c, 128, BN, D / 8, false);  // G^T = K a^T ...
      stage_rows<D>(c, true, Bm + ko, c0, N, BM);
      stage_rows<D>(c, false, Q + qo, q0, N, BN);
      mma3(c, 128, BN, D / 8, true);  // ... + b Q^T
      stage_rows<D>(c, true, V + ko, c0, N, BM);
      stage_rows<D>(c, false, dO + qo, q0, N, BN);
      mma3(c, 64, BN, D / 8, false);  // dP^T = V dO^T
      stage_rows<D>(c, true, C + ko, c0, N, BM);
      mma3(c, 192, BN, D / 8, false);  // H^T = c dO^T
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float s[32], dp[32], g[32], hh[32];
        tld(c, 32 * h, s);
        tld(c, 64 + 32 * h, dp);
        tld(c, 128 + 32 * h, g);
        tld(c, 192 + 32 * h, hh);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int64_t qi = q0 + 32 * h + t;
          const float4 sv = st[32 * h + t];  // (lse, D, E, F) of query qi
          const bool vis = key < N && qi < N && (!causal || (qi >= key && qi <= hi_k));
          const float p = vis ? expf(s[t] * scale - sv.x) : 0.f;
          const float gg = scale * g[t];
          s[t] = p * (gg - sv.z);                                            // dPbar
          g[t] = p * (gg * (dp[t] - sv.y) - sv.z * dp[t] + hh[t] - sv.w);    // Sbar
          dp[t] = p * (dp[t] - sv.y);                                        // dS
        }
        tst(c, 32 * h, s);
        tst(c, 64 + 32 * h, dp);
        tst(c, 128 + 32 * h, g);
      }
      // Block products into the scratch columns 384-447, each added to its accumulator.
      stage_tmem(c, 0);  // dPbar
      stage_rows_t<D>(c, dO + qo, q0, N);
      mma_acc<D>(c, 256, 384, first);  // gV += dPbar^T dO
      stage_tmem(c, 64);  // dS
      stage_rows_t<D>(c, A + qo, q0, N);
      mma_acc<D>(c, 320, 384, first);  // gK += dS^T a
      stage_tmem(c, 128);  // Sbar
      stage_rows_t<D>(c, Q + qo, q0, N);
      mma_acc<D>(c, 320, 384, false);  // gK += Sbar^T Q
      first = false;
    }
  }
  float gv[D], gk[D];
  tld_acc<D>(c, 256, 1.f, gv);
  tld_acc<D>(c, 320, scale, gk);
  if (key < N) {
    store_row<D>(gV + ko + key * D, gv);
    store_row<D>(gK + ko + key * D, gk);
  }
  teardown(c, 512);
}

template <typename Kern>
cudaError_t launch_prep(Kern k, int smem) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

inline int blocks_of(int64_t N, int rows) { return static_cast<int>((N + rows - 1) / rows); }

template <int D>
cudaError_t fwd_t(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse, cudaStream_t st) {
  auto k = f32_fwd_kernel<D>;
  cudaError_t e = launch_prep(k, kSmem);
  if (e != cudaSuccess) return e;
  const int nrb = blocks_of(p.N, BM);
  k<<<static_cast<unsigned>(nrb * p.BH), kThreads, kSmem, st>>>(
      static_cast<const float*>(Q), static_cast<const float*>(K), static_cast<const float*>(V),
      static_cast<float*>(O), lse, static_cast<int>(p.N), nrb, static_cast<int>(p.BH), p.scale, p.causal,
      make_band(p, eff_window(p), false), p.group);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_t(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes, cudaStream_t st) {
  using CF = const float*;
  const int nb = blocks_of(p.N, BM);
  if (passes & 1) {
    auto k = f32_bwd_row_kernel<D>;
    cudaError_t e = launch_prep(k, kSmem);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(nb * p.BH), kThreads, kSmem, st>>>(
        static_cast<CF>(Q), static_cast<CF>(K), static_cast<CF>(V), static_cast<CF>(O), static_cast<CF>(dO), lse,
        static_cast<float*>(dQ), ws, static_cast<int>(p.N), nb, static_cast<int>(p.BH), p.scale, p.causal,
        make_band(p, eff_window(p), false), p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (passes & 2) {
    auto k = f32_bwd_col_kernel<D>;
    cudaError_t e = launch_prep(k, kSmem);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(nb * p.BHkv), kThreads, kSmem, st>>>(
        static_cast<CF>(Q), static_cast<CF>(K), static_cast<CF>(V), static_cast<CF>(dO), ws,
        static_cast<float*>(dK), static_cast<float*>(dV), static_cast<int>(p.N), nb, static_cast<int>(p.BHkv),
        p.scale, p.causal, make_band(p, eff_window(p), true), p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t bob_t(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* lse, const void* a, const void* b, const void* cc, void* gQ, void* gK, void* gV,
                  void* gdO, float4* ws, int passes, cudaStream_t st) {
  using CF = const float*;
  const int nb = blocks_of(p.N, BM);
  if (passes & 1) {
    auto k = f32_bob_row_kernel<D>;
    cudaError_t e = launch_prep(k, kSmemBob);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(nb * p.BH), kThreads, kSmemBob, st>>>(
        static_cast<CF>(Q), static_cast<CF>(K), static_cast<CF>(V), static_cast<CF>(O), static_cast<CF>(dO), lse,
        static_cast<CF>(a), static_cast<CF>(b), static_cast<CF>(cc), static_cast<float*>(gQ),
        static_cast<float*>(gdO), ws, static_cast<int>(p.N), nb, static_cast<int>(p.BH), p.scale, p.causal,
        make_band(p, eff_window(p), false), p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (passes & 2) {
    auto k = f32_bob_col_kernel<D>;
    cudaError_t e = launch_prep(k, kSmemBob);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(nb * p.BHkv), kThreads, kSmemBob, st>>>(
        static_cast<CF>(Q), static_cast<CF>(K), static_cast<CF>(V), static_cast<CF>(dO), static_cast<CF>(a),
        static_cast<CF>(b), static_cast<CF>(cc), ws, static_cast<float*>(gK), static_cast<float*>(gV),
        static_cast<int>(p.N), nb, static_cast<int>(p.BHkv), p.scale, p.causal, make_band(p, eff_window(p), true),
        p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool tc32_supports(int64_t d) { return d == 32 || d == 64; }

cudaError_t tc32_fwd(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse,
                     cudaStream_t st) {
  if (p.d == 32) return fwd_t<32>(p, Q, K, V, O, lse, st);
  if (p.d == 64) return fwd_t<64>(p, Q, K, V, O, lse, st);
  return cudaErrorInvalidValue;
}

cudaError_t tc32_bwd(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes, cudaStream_t st) {
  if (p.d == 32) return bwd_t<32>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st);
  if (p.d == 64) return bwd_t<64>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st);
  return cudaErrorInvalidValue;
}

cudaError_t tc32_bob(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* lse, const void* a, const void* b, const void* c, void* gQ, void* gK, void* gV,
                     void* gdO, float4* ws, int passes, cudaStream_t st) {
  if (p.d == 32) return bob_t<32>(p, Q, K, V, O, dO, lse, a, b, c, gQ, gK, gV, gdO, ws, passes, st);
  if (p.d == 64) return bob_t<64>(p, Q, K, V, O, dO, lse, a, b, c, gQ, gK, gV, gdO, ws, passes, st);
  return cudaErrorInvalidValue;
}

uint32_t tc32_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
