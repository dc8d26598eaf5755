// The tf32 tensor-core engine (tcgen05, kind::tf32): float32 attention at every head dim
// (forward, backward row and column passes, BoB row and column passes), and the bf16
// case the pipelined bf16 kernels do not cover (the BoB at d = 256, with or without GProj).
// The decomposition is the one of the bf16 kernels:
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
//             Sbar = P (G (dP - D) - E dP + H - F);
//   GProj     (bf16 BoB, "FlashAttention bf16 gradient and GProj", "How the zero sum
//             turns into a false gradient"): the products that contract dS see bf16(dS)
//             projected to zero row sum with bf16(P), rho_i = sum_j bf16(dS_ij) /
//             sum_j bf16(P_ij).
//
// Precision: every product A B^T runs as three tf32 products,
//   A B^T ~ A_lo B_hi^T + A_hi B_lo^T + A_hi B_hi^T,
// with x_hi = tf32(x) and x_lo = tf32(x - x_hi) (round to nearest), so each element
// product is exact to about 2^-21 relative (the dropped A_lo B_lo term and the rounding
// of the low parts), accumulated in fp32 in tensor memory; operands that are bf16 input
// rows are exact in tf32 and take one product.  Everything else (softmax, the
// elementwise terms, the states) is fp32 on the CUDA cores with expf.
//
// Structure: one CTA of 128 threads holds 128 rows (queries in row passes, keys in
// column passes), one row per thread and per TMEM lane, and streams blocks of 64
// partner rows.  Each product is one synchronous step: the threads write the two
// operands into 128-byte-swizzled K-major shared-memory tiles (A: 128 rows, B: 64 or
// fewer rows, K up to 64 fp32 in two 128-byte slabs), split into their tf32 high and low
// parts; one warp issues the MMAs and commits them to an mbarrier that every thread
// waits on (bounded).  Operands that are products of the threads' own rows (P, dS, ...)
// are written from registers or copied back from TMEM into the A tile; the transposed
// streamed operands (V^T, K^T, dO^T, ...) are transposed while they are split.  Past
// d = 64 the score-type tiles take the head dim in chunks of 64 and the output columns
// are split over CTAs.  This engine is the precision path (its tolerance is 1e-5, not
// its speed), so the steps are not overlapped.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

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
constexpr int oRho = oSt + BN * 16;   // GProj (bf16 BoB column pass): their 64 coefficients
constexpr int oBar = oRho + BN * 4;
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

// Element access for the two input types: four consecutive elements as floats (bf16
// widens exactly), 32 floats stored (bf16: rounded once, to nearest even).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(tc::bf16_lo(u.x), tc::bf16_hi(u.x), tc::bf16_lo(u.y), tc::bf16_hi(u.y));
}
__device__ __forceinline__ void store32(float* dst, const float (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 32; k += 4) *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
}
__device__ __forceinline__ void store32(__nv_bfloat16* dst, const float (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 32; k += 8)
    *reinterpret_cast<uint4*>(dst + k) = make_uint4(ptx::pack_bf16(v[k], v[k + 1]), ptx::pack_bf16(v[k + 2], v[k + 3]),
                                                    ptx::pack_bf16(v[k + 4], v[k + 5]), ptx::pack_bf16(v[k + 6], v[k + 7]));
}
// Input rows of bf16 are exact in tf32 (8 explicit mantissa bits of 10): their low parts
// are zero, so they are staged without them and multiplied once.
template <typename T>
constexpr bool kExact = std::is_same_v<T, __nv_bfloat16>;
// x rounded to bf16 and widened back (the rounding the GProj reading applies to dS and P).
__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// KW columns [col0, col0 + KW) of R rows (row0 ...) of a row-major array with row
// stride ld, as a K-major tile (K = KW); rows at or past `nrows` are zero.  `a`: the A
// tile (else the B tile).  Every load of the thread is issued before the first store, so
// the L2 round trips overlap.
template <int KW, int R, typename T>
__device__ __forceinline__ void stage_rows(const Ctx& c, bool a, const T* src, int ld, int col0, int64_t row0,
                                           int64_t nrows) {
  constexpr int C4 = KW / 4, IT = R * C4 / kThreads;
  static_assert(R * C4 % kThreads == 0, "staging split");
  uint8_t* hi = c.sm + (a ? oAh : oBh);
  uint8_t* lo = c.sm + (a ? oAl : oBl);
  float4 v[IT];
#pragma unroll
  for (int u = 0; u < IT; ++u) {
    const int idx = threadIdx.x + u * kThreads, row = idx / C4, k = (idx % C4) * 4;
    v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + row < nrows) v[u] = ld4(src + (row0 + row) * ld + col0 + k);
  }
#pragma unroll
  for (int u = 0; u < IT; ++u) {
    const int idx = threadIdx.x + u * kThreads, row = idx / C4, k = (idx % C4) * 4;
    if constexpr (kExact<T>) {
      *reinterpret_cast<float4*>(hi + swz(row, k, R)) = v[u];  // bf16 values are tf32 values
    } else {
      put4(hi, lo, swz(row, k, R), v[u]);
    }
  }
}

// Columns [col0, col0 + KW) of 64 rows (row0 ...) of a row-major array with row stride
// ld, transposed: the B tile of KW rows whose K index is the source row (the products
// whose K is the streamed rows).  Loads first, as above.
template <int KW, typename T>
__device__ __forceinline__ void stage_rows_t(const Ctx& c, const T* src, int ld, int col0, int64_t row0,
                                             int64_t nrows) {
  constexpr int C4 = KW / 4, IT = BN * C4 / kThreads;
  static_assert(BN * C4 % kThreads == 0, "staging split");
  uint8_t* hi = c.sm + oBh;
  uint8_t* lo = c.sm + oBl;
  float4 v[IT];
#pragma unroll
  for (int u = 0; u < IT; ++u) {
    const int idx = threadIdx.x + u * kThreads, srow = idx / C4, col = (idx % C4) * 4;
    v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + srow < nrows) v[u] = ld4(src + (row0 + srow) * ld + col0 + col);
  }
#pragma unroll
  for (int u = 0; u < IT; ++u) {
    const int idx = threadIdx.x + u * kThreads, srow = idx / C4, col = (idx % C4) * 4;
    const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if constexpr (kExact<T>) {
        *reinterpret_cast<float*>(hi + swz(col + q, srow, KW)) = e[q];
      } else {
        put1(hi, lo, swz(col + q, srow, KW), e[q]);
      }
    }
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

// The A tile (K = 64) from 64 TMEM columns of this thread's lane (ROUND: each value
// rounded to bf16 first).
template <bool ROUND = false>
__device__ __forceinline__ void stage_tmem(const Ctx& c, uint32_t col) {
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    float v[32];
    tld(c, col + 32 * h, v);
    if constexpr (ROUND) {
#pragma unroll
      for (int t = 0; t < 32; ++t) v[t] = bf16r(v[t]);
    }
    stage_own(c, 32 * h, v);
  }
}

// TMEM columns [col, col + n) (+)= A B^T over nk K-steps of 8: A = the A tile (128
// rows), B = the B tile (n rows).  Synchronous: returns when the products are done.
// a_exact / b_exact: the operand is exact in tf32 (bf16 input rows: the low part is zero
// and was not staged), so the products with its low part are skipped.
__device__ __forceinline__ void mma3(Ctx& c, uint32_t col, int n, int nk, bool accumulate, bool a_exact = false,
                                     bool b_exact = false) {
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
      uint32_t acc = (accumulate || k > 0) ? 1u : 0u;
      if (!a_exact) {
        ptx::mma_ss_tf32_e(c.tmem + col, dal, dbh, id, acc);
        acc = 1u;
      }
      if (!b_exact) {
        ptx::mma_ss_tf32_e(c.tmem + col, dah, dbl, id, acc);
        acc = 1u;
      }
      ptx::mma_ss_tf32_e(c.tmem + col, dah, dbh, id, acc);
    }
    ptx::mma_commit_e(c.bar);
  }
  const ptx::BoundedWait wait{c.abort_flag, &g_err};
  wait(c.bar, c.phase & 1);
  ++c.phase;
  ptx::tc_fence_after();
}

// A score-type tile: TMEM columns [col, col + 64) (+)= A B^T with A = 128 rows (a0 ...)
// of `a` and B = 64 rows (b0 ...) of `b`, both of row length D, K = D in chunks of 64
// (the last one 32 wide when D = 96), each chunk staged and multiplied in turn.
template <int D, typename T>
__device__ __forceinline__ void tile_product(Ctx& c, uint32_t col, const T* a, int64_t a0, const T* b, int64_t b0,
                                             int N, bool accumulate) {
#pragma unroll 1
  for (int ch = 0; ch < (D + 63) / 64; ++ch) {
    const int k0 = 64 * ch;
    if (D - k0 >= 64) {
      stage_rows<64, BM>(c, true, a, D, k0, a0, N);
      stage_rows<64, BN>(c, false, b, D, k0, b0, N);
      mma3(c, col, BN, 8, accumulate || ch > 0, kExact<T>, kExact<T>);
    } else {
      stage_rows<32, BM>(c, true, a, D, k0, a0, N);
      stage_rows<32, BN>(c, false, b, D, k0, b0, N);
      mma3(c, col, BN, 4, accumulate || ch > 0, kExact<T>, kExact<T>);
    }
  }
}

// Running accumulator (TMEM columns acc .. acc + np) += the block product in the scratch
// columns, in IEEE fp32 on the CUDA cores (first: the accumulator takes the product).
// The tensor core's own accumulation rounds differently from fp32 addition, and its
// error grows with the length of the chain; across blocks the sums are kept here.
__device__ __forceinline__ void add_into(const Ctx& c, uint32_t acc, uint32_t scr, int np, bool first) {
#pragma unroll 1
  for (int h = 0; h < np / 32; ++h) {
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
// An output-type product for this CTA's output columns [p0, p0 + np): the A tile (K =
// the 64 streamed rows) times columns p0 .. p0 + np of the streamed rows (b0 ...) of `b`
// (row length ld), into the scratch columns, then added to the accumulator.
template <typename T>
__device__ __forceinline__ void out_product(Ctx& c, uint32_t acc, uint32_t scr, const T* b, int ld, int p0, int np,
                                            int64_t b0, int N, bool first) {
  if (np == 64) {
    stage_rows_t<64>(c, b, ld, p0, b0, N);
  } else {
    stage_rows_t<32>(c, b, ld, p0, b0, N);
  }
  mma3(c, scr, np, BN / 8, false, false, kExact<T>);
  add_into(c, acc, scr, np, first);
}

// dot(x_i, y_i) over a row of D elements, in fp32.
template <int D, typename T>
__device__ __forceinline__ float row_dot(const T* x, const T* y) {
  float acc = 0.f;
#pragma unroll 4
  for (int k = 0; k < D; k += 4) {
    const float4 a = ld4(x + k), b = ld4(y + k);
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    acc = fmaf(a.w, b.w, acc);
  }
  return acc;
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

// Output columns are split over parts of PW (CTAs of one block of rows differ only in
// the part they accumulate and write; each computes the whole score-type tiles).
constexpr int parts_of(int D, int PW) { return (D + PW - 1) / PW; }
struct Where {
  int slice, blk, p0, np;  // slice, block of rows (heaviest first where it matters), output columns
};
template <int D, int PW>
__device__ __forceinline__ Where where(int nslices, int nblk, bool reverse) {
  const int x = static_cast<int>(blockIdx.x);
  const int part = x % parts_of(D, PW);
  const tc::Order o = tc::grid_order_at(x / parts_of(D, PW), nslices, nblk);
  const int p0 = PW * part;
  return Where{o.bh, reverse ? nblk - 1 - o.k : o.k, p0, min(PW, D - p0)};
}

// ------------------------------------------------------------------ forward
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_fwd_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, T* __restrict__ O,
                   float* __restrict__ lse, int N, int nrb, int BH, float scale, int causal, Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  Ctx c = setup(sm, 128);  // S / P 0-63, P V 64-127
  const Where w = where<D, 64>(BH, nrb, true);
  const int bh = w.slice, rb = w.blk, kvh = bh / G;
  const int64_t i = static_cast<int64_t>(rb) * BM + threadIdx.x;
  const T* q = Q + static_cast<size_t>(bh) * N * D;
  const T* k = K + static_cast<size_t>(kvh) * N * D;
  const T* v = V + static_cast<size_t>(kvh) * N * D;
  const int lo_i = causal ? bd.row_lo(bh, i) : 0;
  const RowRange rr = key_blocks(rb, N, causal, bd, bh);
  float m = -INFINITY, l = 0.f, o[64];  // this part's np <= 64 output columns
#pragma unroll
  for (int t = 0; t < 64; ++t) o[t] = 0.f;
  for (int kb = rr.k0; kb < rr.k1; ++kb) {
    tile_product<D>(c, 0, q, static_cast<int64_t>(rb) * BM, k, static_cast<int64_t>(kb) * BN, N, false);  // S = Q K^T
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
    if (w.np == 64) {
      stage_rows_t<64>(c, v, D, w.p0, static_cast<int64_t>(kb) * BN, N);
    } else {
      stage_rows_t<32>(c, v, D, w.p0, static_cast<int64_t>(kb) * BN, N);
    }
    mma3(c, 64, w.np, BN / 8, false);  // P V, this part's columns
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (32 * h < w.np) {
        float pv[32];
        tld(c, 64 + 32 * h, pv);
#pragma unroll
        for (int t = 0; t < 32; ++t) o[32 * h + t] = o[32 * h + t] * alpha + pv[t];
      }
    }
  }
  if (i < N) {
    const float inv = 1.f / l;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (32 * h < w.np) {
        float out[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) out[t] = o[32 * h + t] * inv;
        store32(O + (static_cast<size_t>(bh) * N + i) * D + w.p0 + 32 * h, out);
      }
    }
    if (w.p0 == 0) lse[static_cast<size_t>(bh) * N + i] = m + logf(l);
  }
  teardown(c, 128);
}

// --------------------------------------------------------- backward, rows
// dQ = s dS K with dS in fp32 (GProj, a bf16 rounding remedy, does not apply).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bwd_row_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                       const T* __restrict__ O, const T* __restrict__ dO, const float* __restrict__ lse,
                       T* __restrict__ dQ, float4* __restrict__ ws, int N, int nrb, int BH, float scale, int causal,
                       Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  Ctx c = setup(sm, 256);  // S 0-63, dP 64-127, dQ 128-191 (this part's columns)
  const Where w = where<D, 64>(BH, nrb, true);
  const int bh = w.slice, rb = w.blk, kvh = bh / G;
  const int64_t i = static_cast<int64_t>(rb) * BM + threadIdx.x, r0 = static_cast<int64_t>(rb) * BM;
  const size_t qo = static_cast<size_t>(bh) * N * D, ko = static_cast<size_t>(kvh) * N * D;
  const int lo_i = causal ? bd.row_lo(bh, i) : 0;
  float Di = 0.f, Li = 0.f;
  if (i < N) {
    Di = row_dot<D>(dO + qo + i * D, O + qo + i * D);
    Li = lse[static_cast<size_t>(bh) * N + i];
  }
  const RowRange rr = key_blocks(rb, N, causal, bd, bh);
  for (int kb = rr.k0; kb < rr.k1; ++kb) {
    const int64_t k0 = static_cast<int64_t>(kb) * BN;
    tile_product<D>(c, 0, Q + qo, r0, K + ko, k0, N, false);    // S = Q K^T
    tile_product<D>(c, 64, dO + qo, r0, V + ko, k0, N, false);  // dP = dO V^T
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float s[32], dp[32];
      tld(c, 32 * h, s);
      tld(c, 64 + 32 * h, dp);
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int64_t key = k0 + 32 * h + t;
        const bool vis = i < N && key < N && (!causal || (key <= i && key >= lo_i));
        const float p = vis ? expf(s[t] * scale - Li) : 0.f;
        s[t] = p * (dp[t] - Di);
      }
      stage_own(c, 32 * h, s);
    }
    out_product(c, 128, 0, K + ko, D, w.p0, w.np, k0, N, kb == rr.k0);  // dQ += dS K (scratch: the read S)
  }
#pragma unroll 1
  for (int h = 0; h < w.np / 32; ++h) {
    float g[32];
    tld(c, 128 + 32 * h, g);
#pragma unroll
    for (int t = 0; t < 32; ++t) g[t] *= scale;
    if (i < N) store32(dQ + qo + i * D + w.p0 + 32 * h, g);
  }
  if (i < N && w.p0 == 0) ws[static_cast<size_t>(bh) * N + i] = make_float4(Li, Di, 0.f, 0.f);
  teardown(c, 256);
}

// ------------------------------------------------------- backward, columns
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bwd_col_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                       const T* __restrict__ dO, const float4* __restrict__ ws, T* __restrict__ dK, T* __restrict__ dV,
                       int N, int nkb, int BHkv, float scale, int causal, Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  Ctx c = setup(sm, 256);  // S^T / P^T 0-63, dP^T / dS^T 64-127, dV 128-191, dK 192-255
  const Where w = where<D, 64>(BHkv, nkb, false);
  const int kvh = w.slice, kb = w.blk;
  const int64_t key = static_cast<int64_t>(kb) * BM + threadIdx.x, c0 = static_cast<int64_t>(kb) * BM;
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
      tile_product<D>(c, 0, K + ko, c0, Q + qo, q0, N, false);    // S^T = K Q^T (mma3's barrier publishes the states)
      tile_product<D>(c, 64, V + ko, c0, dO + qo, q0, N, false);  // dP^T = V dO^T
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
          dp[t] = p * (dp[t] - sv.y);
          s[t] = p;
        }
        stage_own(c, 32 * h, s);  // P^T
        tst(c, 64 + 32 * h, dp);
      }
      out_product(c, 128, 0, dO + qo, D, w.p0, w.np, q0, N, first);  // dV += P^T dO (scratch: the read S^T)
      stage_tmem(c, 64);
      out_product(c, 192, 0, Q + qo, D, w.p0, w.np, q0, N, first);   // dK += dS^T Q
      first = false;
    }
  }
#pragma unroll 1
  for (int h = 0; h < w.np / 32; ++h) {
    float gv[32], gk[32];
    tld(c, 128 + 32 * h, gv);
    tld(c, 192 + 32 * h, gk);
#pragma unroll
    for (int t = 0; t < 32; ++t) gk[t] *= scale;
    if (key < N) {
      store32(dV + ko + key * D + w.p0 + 32 * h, gv);
      store32(dK + ko + key * D + w.p0 + 32 * h, gk);
    }
  }
  teardown(c, 256);
}

// ------------------------------------------------------------------ BoB, rows
// GP (bf16 inputs): Y's dS b product sees bf16(dS), P^ b = sum_j bf16(P_ij) b_j is
// accumulated beside it and gQ -= s rho P^ b with rho_i = sum_j bf16(dS_ij) / sum_j
// bf16(P_ij); rho goes to rho_ws (one float per row, slice pitch N).  The GP CTAs take
// 32 output columns each, so that the fifth accumulator fits TMEM.
template <typename T, int D, bool GP>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bob_row_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                       const T* __restrict__ O, const T* __restrict__ dO, const float* __restrict__ lse,
                       const T* __restrict__ A, const T* __restrict__ Bm, const T* __restrict__ C, T* __restrict__ gQ,
                       T* __restrict__ gdO, float4* __restrict__ ws, float* __restrict__ rho_ws, int N, int nrb,
                       int BH, float scale, int causal, Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  constexpr int PW = GP ? 32 : 64;  // output columns per CTA
  // TMEM: S / P 0, dP / dS 64, G / PG 128, H / W 192, and this part's X, Y, Z, U (and with
  // GP P^ b and the scratch) at 256 + PW j.
  constexpr uint32_t cX = 256, cY = 256 + PW, cZ = 256 + 2 * PW, cU = 256 + 3 * PW, cPb = 256 + 4 * PW;
  constexpr uint32_t cScr = GP ? 256 + 5 * PW : 0;
  Ctx c = setup(sm, 512);
  const Where w = where<D, PW>(BH, nrb, true);
  const int bh = w.slice, rb = w.blk, kvh = bh / G;
  const int64_t i = static_cast<int64_t>(rb) * BM + threadIdx.x, r0 = static_cast<int64_t>(rb) * BM;
  const size_t qo = static_cast<size_t>(bh) * N * D, ko = static_cast<size_t>(kvh) * N * D;
  const int lo_i = causal ? bd.row_lo(bh, i) : 0;
  // E, F' = sum W, and the row sums of P and dS as the products see them (fp32); r, sp:
  // the GProj sums of bf16(dS) and bf16(P).
  float Di = 0.f, Li = 0.f, E = 0.f, Fp = 0.f, sP = 0.f, sdS = 0.f, r = 0.f, sp = 0.f;
  if (i < N) {
    Di = row_dot<D>(dO + qo + i * D, O + qo + i * D);
    Li = lse[static_cast<size_t>(bh) * N + i];
  }
  const RowRange rr = key_blocks(rb, N, causal, bd, bh);
  for (int kb = rr.k0; kb < rr.k1; ++kb) {
    const int64_t k0 = static_cast<int64_t>(kb) * BN;
    const bool acc = kb > rr.k0;
    tile_product<D>(c, 0, Q + qo, r0, K + ko, k0, N, false);     // S = Q K^T
    tile_product<D>(c, 128, Q + qo, r0, Bm + ko, k0, N, false);  // G = Q b^T ...
    tile_product<D>(c, 128, A + qo, r0, K + ko, k0, N, true);    // ... + a K^T
    tile_product<D>(c, 64, dO + qo, r0, V + ko, k0, N, false);   // dP = dO V^T
    tile_product<D>(c, 192, dO + qo, r0, C + ko, k0, N, false);  // H = dO c^T
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
        const float wv = gg * ds + p * hh[t];
        E += pg;
        Fp += wv;
        sP += p;
        sdS += ds;
        if constexpr (GP) {
          r += bf16r(ds);
          sp += bf16r(p);
        }
        s[t] = p;
        dp[t] = ds;
        g[t] = pg;
        hh[t] = wv;
      }
      tst(c, 32 * h, s);
      tst(c, 64 + 32 * h, dp);
      tst(c, 128 + 32 * h, g);
      tst(c, 192 + 32 * h, hh);
    }
    // Block products into the scratch columns (0-63 without GP: P, once in the A tile,
    // is not read from TMEM again; 416-447 with GP, where P is read again rounded), each
    // added to its accumulator.
    stage_tmem(c, 0);  // P
    out_product(c, cX, cScr, C + ko, D, w.p0, w.np, k0, N, !acc);   // X += P c
    out_product(c, cU, cScr, K + ko, D, w.p0, w.np, k0, N, !acc);   // U += P K
    stage_tmem(c, 128);  // P G
    out_product(c, cX, cScr, V + ko, D, w.p0, w.np, k0, N, false);  // X += (P G) V
    stage_tmem(c, 64);  // dS
    out_product(c, cZ, cScr, K + ko, D, w.p0, w.np, k0, N, !acc);   // Z += dS K
    if constexpr (GP) stage_tmem<true>(c, 64);  // bf16(dS)
    out_product(c, cY, cScr, Bm + ko, D, w.p0, w.np, k0, N, !acc);  // Y += dS b
    stage_tmem(c, 192);  // W
    out_product(c, cY, cScr, K + ko, D, w.p0, w.np, k0, N, false);  // Y += W K
    if constexpr (GP) {
      stage_tmem<true>(c, 0);  // bf16(P)
      out_product(c, cPb, cScr, Bm + ko, D, w.p0, w.np, k0, N, !acc);  // P^ b
    }
  }
  const float rho = GP ? r / sp : 0.f;
  // The correction of the K-multiplied terms takes F' as the products see it, (F' - E sum
  // dS) / sum P, so that the row W - E dS - F' P they effectively contract sums to zero
  // (the exact row does: sum dS = 0, sum P = 1).  With bf16 O, D and with it sum dS are
  // off by the rounding of O, and a large mean key would multiply that residual.
  const float Fq = (Fp - E * sdS) / sP;
#pragma unroll 1
  for (int h = 0; h < w.np / 32; ++h) {  // 32 output columns at a time
    float x[32], y[32], z[32], u[32];
    tld(c, cX + 32 * h, x);
    tld(c, cY + 32 * h, y);
    tld(c, cZ + 32 * h, z);
    tld(c, cU + 32 * h, u);
    if constexpr (GP) {
      float pb[32];
      tld(c, cPb + 32 * h, pb);
#pragma unroll
      for (int t = 0; t < 32; ++t) y[t] -= rho * pb[t];
    }
    if (i < N) {
      const T* orow = O + qo + i * D + w.p0 + 32 * h;
#pragma unroll
      for (int t = 0; t < 32; t += 4) {
        const float4 o4 = ld4(orow + t);
        const float ov[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[t + e] = x[t + e] - E * ov[e];                               // gdO
          y[t + e] = scale * (y[t + e] - E * z[t + e] - Fq * u[t + e]);  // gQ
        }
      }
      store32(gdO + qo + i * D + w.p0 + 32 * h, x);
      store32(gQ + qo + i * D + w.p0 + 32 * h, y);
    }
  }
  if (i < N && w.p0 == 0) {
    ws[static_cast<size_t>(bh) * N + i] = make_float4(Li, Di, E, Fp - E * Di);
    if constexpr (GP) rho_ws[static_cast<size_t>(bh) * N + i] = rho;
  }
  teardown(c, 512);
}

// --------------------------------------------------------------- BoB, columns
// GP (bf16 inputs): gK's dS^T a product sees the projected bf16(dS) - rho_i bf16(P)
// (rho from rho_ws).
template <typename T, int D, bool GP>
__global__ void __launch_bounds__(kThreads, 1)
    f32_bob_col_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                       const T* __restrict__ dO, const T* __restrict__ A, const T* __restrict__ Bm,
                       const T* __restrict__ C, const float4* __restrict__ ws, const float* __restrict__ rho_ws,
                       T* __restrict__ gK, T* __restrict__ gV, int N, int nkb, int BHkv, float scale, int causal,
                       Band bd, int G) {
  extern __shared__ __align__(1024) uint8_t sm[];
  // TMEM: S^T / dPbar 0, dP^T / dS 64, G^T / Sbar 128, H^T 192, this part's gV 256 and
  // gK 320, scratch 384.
  Ctx c = setup(sm, 512);
  const Where w = where<D, 64>(BHkv, nkb, false);
  const int kvh = w.slice, kb = w.blk;
  const int64_t key = static_cast<int64_t>(kb) * BM + threadIdx.x, c0 = static_cast<int64_t>(kb) * BM;
  const size_t ko = static_cast<size_t>(kvh) * N * D;
  const int hi_k = causal ? bd.key_hi(kvh, key) : N - 1;
  const RowRange qr = query_blocks(kb, N, causal, bd, kvh);
  const float4* st = reinterpret_cast<const float4*>(sm + oSt);
  const float* rs = reinterpret_cast<const float*>(sm + oRho);
  bool first = true;
  for (int hq = kvh * G; hq < (kvh + 1) * G; ++hq) {
    const size_t qo = static_cast<size_t>(hq) * N * D;
    for (int qb = qr.k0; qb < qr.k1; ++qb) {
      const int64_t q0 = static_cast<int64_t>(qb) * BN;
      if (threadIdx.x < BN) {
        const int64_t qi = q0 + threadIdx.x;
        reinterpret_cast<float4*>(sm + oSt)[threadIdx.x] =
            qi < N ? ws[static_cast<size_t>(hq) * N + qi] : make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (GP) reinterpret_cast<float*>(sm + oRho)[threadIdx.x] = qi < N ? rho_ws[static_cast<size_t>(hq) * N + qi] : 0.f;
      }
      tile_product<D>(c, 0, K + ko, c0, Q + qo, q0, N, false);     // S^T = K Q^T (mma3's barrier publishes the states)
      tile_product<D>(c, 128, K + ko, c0, A + qo, q0, N, false);   // G^T = K a^T ...
      tile_product<D>(c, 128, Bm + ko, c0, Q + qo, q0, N, true);   // ... + b Q^T
      tile_product<D>(c, 64, V + ko, c0, dO + qo, q0, N, false);   // dP^T = V dO^T
      tile_product<D>(c, 192, C + ko, c0, dO + qo, q0, N, false);  // H^T = c dO^T
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
          s[t] = p * (gg - sv.z);                                          // dPbar
          g[t] = p * (gg * (dp[t] - sv.y) - sv.z * dp[t] + hh[t] - sv.w);  // Sbar
          const float ds = p * (dp[t] - sv.y);                             // dS
          dp[t] = GP ? bf16r(ds) - rs[32 * h + t] * bf16r(p) : ds;
        }
        tst(c, 32 * h, s);
        tst(c, 64 + 32 * h, dp);
        tst(c, 128 + 32 * h, g);
      }
      // Block products into the scratch columns 384-447, each added to its accumulator.
      stage_tmem(c, 0);  // dPbar
      out_product(c, 256, 384, dO + qo, D, w.p0, w.np, q0, N, first);  // gV += dPbar^T dO
      stage_tmem(c, 64);  // dS (GP: projected)
      out_product(c, 320, 384, A + qo, D, w.p0, w.np, q0, N, first);   // gK += dS^T a
      stage_tmem(c, 128);  // Sbar
      out_product(c, 320, 384, Q + qo, D, w.p0, w.np, q0, N, false);   // gK += Sbar^T Q
      first = false;
    }
  }
#pragma unroll 1
  for (int h = 0; h < w.np / 32; ++h) {
    float gv[32], gk[32];
    tld(c, 256 + 32 * h, gv);
    tld(c, 320 + 32 * h, gk);
#pragma unroll
    for (int t = 0; t < 32; ++t) gk[t] *= scale;
    if (key < N) {
      store32(gV + ko + key * D + w.p0 + 32 * h, gv);
      store32(gK + ko + key * D + w.p0 + 32 * h, gk);
    }
  }
  teardown(c, 512);
}

template <typename Kern>
cudaError_t launch_prep(Kern k, int smem) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

inline int blocks_of(int64_t N, int rows) { return static_cast<int>((N + rows - 1) / rows); }
inline unsigned grid_of(int nblk, int64_t slices, int parts) {
  return static_cast<unsigned>(static_cast<int64_t>(nblk) * slices * parts);
}

template <typename T, int D>
cudaError_t fwd_t(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse, cudaStream_t st) {
  auto k = f32_fwd_kernel<T, D>;
  cudaError_t e = launch_prep(k, kSmem);
  if (e != cudaSuccess) return e;
  const int nrb = blocks_of(p.N, BM);
  k<<<grid_of(nrb, p.BH, parts_of(D, 64)), kThreads, kSmem, st>>>(
      static_cast<const T*>(Q), static_cast<const T*>(K), static_cast<const T*>(V), static_cast<T*>(O), lse,
      static_cast<int>(p.N), nrb, static_cast<int>(p.BH), p.scale, p.causal, make_band(p, eff_window(p), false),
      p.group);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_t(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes, cudaStream_t st) {
  using CT = const T*;
  const int nb = blocks_of(p.N, BM);
  if (passes & 1) {
    auto k = f32_bwd_row_kernel<T, D>;
    cudaError_t e = launch_prep(k, kSmem);
    if (e != cudaSuccess) return e;
    k<<<grid_of(nb, p.BH, parts_of(D, 64)), kThreads, kSmem, st>>>(
        static_cast<CT>(Q), static_cast<CT>(K), static_cast<CT>(V), static_cast<CT>(O), static_cast<CT>(dO), lse,
        static_cast<T*>(dQ), ws, static_cast<int>(p.N), nb, static_cast<int>(p.BH), p.scale, p.causal,
        make_band(p, eff_window(p), false), p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (passes & 2) {
    auto k = f32_bwd_col_kernel<T, D>;
    cudaError_t e = launch_prep(k, kSmem);
    if (e != cudaSuccess) return e;
    k<<<grid_of(nb, p.BHkv, parts_of(D, 64)), kThreads, kSmem, st>>>(
        static_cast<CT>(Q), static_cast<CT>(K), static_cast<CT>(V), static_cast<CT>(dO), ws, static_cast<T*>(dK),
        static_cast<T*>(dV), static_cast<int>(p.N), nb, static_cast<int>(p.BHkv), p.scale, p.causal,
        make_band(p, eff_window(p), true), p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T, int D, bool GP>
cudaError_t bob_t(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* lse, const void* a, const void* b, const void* cc, void* gQ, void* gK, void* gV,
                  void* gdO, float4* ws, float* rho_ws, int passes, cudaStream_t st) {
  using CT = const T*;
  const int nb = blocks_of(p.N, BM);
  if (passes & 1) {
    auto k = f32_bob_row_kernel<T, D, GP>;
    cudaError_t e = launch_prep(k, kSmemBob);
    if (e != cudaSuccess) return e;
    k<<<grid_of(nb, p.BH, parts_of(D, GP ? 32 : 64)), kThreads, kSmemBob, st>>>(
        static_cast<CT>(Q), static_cast<CT>(K), static_cast<CT>(V), static_cast<CT>(O), static_cast<CT>(dO), lse,
        static_cast<CT>(a), static_cast<CT>(b), static_cast<CT>(cc), static_cast<T*>(gQ), static_cast<T*>(gdO), ws,
        rho_ws, static_cast<int>(p.N), nb, static_cast<int>(p.BH), p.scale, p.causal,
        make_band(p, eff_window(p), false), p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (passes & 2) {
    auto k = f32_bob_col_kernel<T, D, GP>;
    cudaError_t e = launch_prep(k, kSmemBob);
    if (e != cudaSuccess) return e;
    k<<<grid_of(nb, p.BHkv, parts_of(D, 64)), kThreads, kSmemBob, st>>>(
        static_cast<CT>(Q), static_cast<CT>(K), static_cast<CT>(V), static_cast<CT>(dO), static_cast<CT>(a),
        static_cast<CT>(b), static_cast<CT>(cc), ws, rho_ws, static_cast<T*>(gK), static_cast<T*>(gV),
        static_cast<int>(p.N), nb, static_cast<int>(p.BHkv), p.scale, p.causal, make_band(p, eff_window(p), true),
        p.group);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// float32 at every head dim; bf16 only at d = 256 (the BoB, which has no bf16 kernel there).
template <typename F>
cudaError_t with_case(const Problem& p, F&& f) {
  if (p.dtype == ATTN_BF16) {
    if (p.d == 256) return f(__nv_bfloat16{}, std::integral_constant<int, 256>{});
    return cudaErrorInvalidValue;
  }
  switch (p.d) {
    case 32: return f(float{}, std::integral_constant<int, 32>{});
    case 64: return f(float{}, std::integral_constant<int, 64>{});
    case 96: return f(float{}, std::integral_constant<int, 96>{});
    case 128: return f(float{}, std::integral_constant<int, 128>{});
    case 256: return f(float{}, std::integral_constant<int, 256>{});
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool tc32_supports(int64_t d) { return d == 32 || d == 64 || d == 96 || d == 128 || d == 256; }

cudaError_t tc32_fwd(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse,
                     cudaStream_t st) {
  return with_case(p, [&](auto t, auto dd) {
    using T = decltype(t);
    if constexpr (std::is_same_v<T, float>) return fwd_t<T, dd()>(p, Q, K, V, O, lse, st);
    return cudaErrorInvalidValue;  // the bf16 forward has its own kernels at every d
  });
}

cudaError_t tc32_bwd(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes, cudaStream_t st) {
  return with_case(p, [&](auto t, auto dd) {
    using T = decltype(t);
    if constexpr (std::is_same_v<T, float>) return bwd_t<T, dd()>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st);
    return cudaErrorInvalidValue;  // the bf16 backward has its own kernels at every d
  });
}

cudaError_t tc32_bob(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* lse, const void* a, const void* b, const void* c, void* gQ, void* gK, void* gV,
                     void* gdO, bool gproj, float4* ws, int passes, cudaStream_t st) {
  float* rho_ws = reinterpret_cast<float*>(bob_rho_region(ws, p));
  return with_case(p, [&](auto t, auto dd) {
    using T = decltype(t);
    if constexpr (std::is_same_v<T, __nv_bfloat16>) {
      if (gproj) return bob_t<T, dd(), true>(p, Q, K, V, O, dO, lse, a, b, c, gQ, gK, gV, gdO, ws, rho_ws, passes, st);
    }
    return bob_t<T, dd(), false>(p, Q, K, V, O, dO, lse, a, b, c, gQ, gK, gV, gdO, ws, nullptr, passes, st);
  });
}

uint32_t tc32_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
