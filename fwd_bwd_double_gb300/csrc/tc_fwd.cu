// bf16 causal attention forward on sm_103a: TMA-fed shared-memory tiles, tcgen05
// MMAs accumulating in tensor memory, online softmax on CUDA cores.
//
// "Flash attention for trading models", sections "The Flash Attention algorithm"
// and "Online softmax recurrence": one CTA owns a block of BM = 128 query rows and
// streams key/value blocks of BN = 128 keys (only blocks j <= i: section "Causal
// masking ...": future blocks are never loaded).  Per block:
//   S = Q K_j^T            tcgen05.mma, A = Q and B = K_j from shared memory,
//                          accumulator in TMEM (128 lanes = query rows)
//   m_new = max(m, rowmax S); p = 2^((S - m_new) s log2 e)   (subtract, then scale:
//                          "FlashAttention bf16 gradient and GProj", "Why the error
//                          appears late", so the row max maps to exactly 1)
//   O <- O 2^((m - m_new) s log2 e) only for rows whose max moved (FA2's deferred
//                          rescaling; O stays unnormalised until the end)
//   O += P V_j             tcgen05.mma, A = P (bf16, two values per 32-bit TMEM
//                          column, lane = query row), B = V_j (MN-major, shared)
// and at the end O / l is written once and lse = m s + ln l.
//
// Warp roles (192 threads): warps 0-3 own TMEM lanes 0-127, one query row per
// thread (softmax, rescale, epilogue); warp 4 issues TMA loads (Q once, K/V
// through a 3-stage ring); warp 5 allocates TMEM and issues the MMAs.  The softmax
// warps copy S_j into registers and release it at once (`s_consumed`), so
// S_{j+1} = Q K_{j+1}^T runs on the tensor pipe while they exponentiate S_j; P_j
// is written into its TMEM columns, and O rescaled, only after P_{j-1} V_{j-1}
// has finished (`pv_done`).  With d = 64 two CTAs fit on an SM (256 TMEM columns
// each), so one CTA's softmax also overlaps the other's MMAs.  At d = 256 (224 threads)
// K and V have a 128-key buffer each and their own TMA warps (4: K, 6: V): K_{j+1} loads
// as soon as S_j is done (`k_empty`), V_{j+1} as soon as P_j V_j is (`empty`), so the
// 128-key blocks fit beside the 64 KB Q tile.
//
// The PB instance serves the GProj form of the backward over backward: with the
// stored log-sum-exp L and the cotangent b in place of V it accumulates
// Pb_i = sum_j P^_ij b_j, P^_ij = bf16(2^(S_ij s log2 e - L_i log2 e)), which is the
// probability row the BoB row pass rounds for its products, formed by the same
// operations on the same S (Q K^T over the same K-steps).  No running max, no
// rescaling, no normalisation; Pb is written in fp32.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fbd {
namespace {

__device__ unsigned int g_err = 0;

constexpr int BM = 128;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Layout {
  // Key blocks of BN = 128 keys.  Up to d = 128 they come through a ring of NS = 3 stages
  // of K and V (2 CTAs per SM at d = 64 still fit).  At d = 256 (SPLIT) the Q tile alone is
  // 64 KB: K and V have one 128-key buffer each, reloaded independently as soon as the
  // product reading it is done (K after S_j, V after P_j V_j), by a TMA warp each.
  static constexpr bool SPLIT = D > 128;
  static constexpr int BN = 128;
  static constexpr int NS = SPLIT ? 1 : 3;
  static constexpr int kThreads = SPLIT ? 224 : 192;  // 4 softmax warps, TMA, MMA (+ the V loader)
  static constexpr int kQ = BM * D * 2;   // bytes of the Q tile
  static constexpr int kKV = BN * D * 2;  // bytes of one K (or V) tile
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + kQ;
  static constexpr int oV = oK + NS * kKV;
  static constexpr int oBar = oV + NS * kKV;
  static constexpr int bytes = oBar + 128;
  // TMEM columns: S fp32 [0, BN), P bf16 pairs [BN, BN + BN/2), O fp32 after them (D).
  static constexpr int kTmemCols = (BN + BN / 2 + D <= 256) ? 256 : 512;
};

// Shared-memory descriptor of a K-major operand tile stored as 64-element
// (128-byte) column slabs of `rows` rows each, advanced to K-step k (16 elements).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int rows, int k) {
  return ptx::sdesc_sw128(base + (k >> 2) * rows * 128 + (k & 3) * 32, 16, 1024);
}
// MN-major operand (rows = K index, 64-element slabs along MN of `rows` rows),
// advanced to K-step k (16 rows).
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int rows, int k) {
  return ptx::sdesc_sw128(base + k * 16 * 128, rows * 128, 1024);
}

// WIN: a banded causal mask is in force (bd: the sliding window and/or the document
// bounds); the instances without it carry none of its arithmetic.
template <int D, bool PB, bool WIN>
__global__ void __launch_bounds__(Layout<D>::kThreads, (D == 64 ? 2 : 1))
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O, float* __restrict__ lse,
               const float* __restrict__ lse_in, float* __restrict__ pb, int N, int nrb, int BH, float scale,
               float scale_log2, int causal, Band bd, int G, int dv) {
  using Lay = Layout<D>;
  constexpr int BN = Lay::BN, NS = Lay::NS;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
  uint64_t* q_full = bars + 0;
  uint64_t* full = bars + 1;            // [NS]
  uint64_t* empty = bars + 1 + NS;      // [NS]
  uint64_t* s_full = bars + 1 + 2 * NS;
  uint64_t* p_ready = s_full + 1;     // P_j in TMEM and O rescaled
  uint64_t* o_full = s_full + 2;
  uint64_t* s_consumed = s_full + 3;  // S_j copied into the softmax registers
  uint64_t* pv_done = s_full + 4;     // P_j V_j finished: P columns and O free
  // SPLIT: full[0] = K_j loaded, empty[0] = P_j V_j done (the V buffer free), and
  uint64_t* v_full = s_full + 5;      // V_j loaded
  uint64_t* k_empty = s_full + 6;     // S_j done (the K buffer free)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + (Lay::SPLIT ? 7 : 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Order ord = tc::grid_order(BH, nrb);
  const int bh = ord.bh;
  const int kvh = bh / G;          // the key/value slice this query slice reads
  const int rb = nrb - 1 - ord.k;  // heaviest row blocks first (within a group of slices)
  // Key blocks this row block sees: j0 + j for j < nkv.  bd: the banded causal mask (row i
  // sees the keys bd.row_lo(i) <= k <= i: the window and/or the document bounds).
  const int j0 = (WIN && causal) ? bd.row_lo(bh, rb * BM) / BN : 0;
  // the lowest key a row of the block sees at the block's last row (rows at or past N
  // looked up at N - 1): blocks starting below it hold keys some row does not see
  const int lo_last = (WIN && causal) ? bd.row_lo(bh, min(rb * BM + BM - 1, N - 1)) : 0;
  const int nkv = (BN == BM ? (causal ? rb + 1 : nrb) : (causal ? ((rb + 1) * BM + BN - 1) / BN : (N + BN - 1) / BN)) - j0;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(p_ready, 128);
    ptx::mbar_init(o_full, 1);
    ptx::mbar_init(s_consumed, 128);
    ptx::mbar_init(pv_done, 1);
    if constexpr (Lay::SPLIT) {
      ptx::mbar_init(v_full, 1);
      ptx::mbar_init(k_empty, 1);
    }
    // The swizzled operand layout needs 1024-byte aligned tiles.
    *abort_flag = (ptx::smem_u32(sm) & 1023u) ? 1 : 0;
    if (*abort_flag) atomicOr(&g_err, FBD_ERR_TIMEOUT);
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(tmem_slot, Lay::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;                 // S accumulator
  const uint32_t tP = tmem + BN;            // P, bf16 A operand of P V
  const uint32_t tO = tmem + BN + BN / 2;   // O accumulator
  const ptx::BoundedWait wait{abort_flag, &g_err};
  const bool ok = *abort_flag == 0;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ok) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::mbar_expect_tx(q_full, Lay::kQ);
      for (int c = 0; c < D / 64; ++c) ptx::tma_load_3d(sm + Lay::oQ + c * BM * 128, &tmQ, q_full, c * 64, rb * BM, bh);
      if constexpr (Lay::SPLIT) {  // K only (the V loader is warp 6)
        for (int j = 0; j < nkv; ++j) {
          if (j >= 1) wait(k_empty, (j - 1) & 1);
          ptx::mbar_expect_tx(&full[0], Lay::kKV);
          for (int c = 0; c < D / 64; ++c)
            ptx::tma_load_3d(sm + Lay::oK + c * BN * 128, &tmK, &full[0], c * 64, (j0 + j) * BN, kvh);
        }
        if (nkv > 0) wait(k_empty, (nkv - 1) & 1);
      } else {
        for (int j = 0; j < nkv; ++j) {
          const int s = j % NS;
          if (j >= NS) wait(&empty[s], ((j / NS) - 1) & 1);
          ptx::mbar_expect_tx(&full[s], 2 * Lay::kKV);
          for (int c = 0; c < D / 64; ++c) {
            ptx::tma_load_3d(sm + Lay::oK + s * Lay::kKV + c * BN * 128, &tmK, &full[s], c * 64, (j0 + j) * BN, kvh);
            ptx::tma_load_3d(sm + Lay::oV + s * Lay::kKV + c * BN * 128, &tmV, &full[s], c * 64, (j0 + j) * BN, kvh);
          }
        }
        // Drain: the last NS stages must have been consumed before the CTA exits.
        for (int j = (nkv > NS ? nkv - NS : 0); j < nkv; ++j) wait(&empty[j % NS], (j / NS) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idS = ptx::idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idO = ptx::idesc_bf16(BM, D, 0, 1);
      // Descriptors at K-step 0 of stage 0, stepped with one add per MMA.
      const uint64_t dQ = kmajor_desc(ptx::smem_u32(sm + Lay::oQ), BM, 0);
      const uint64_t dK = kmajor_desc(ptx::smem_u32(sm + Lay::oK), BN, 0);
      const uint64_t dV = mnmajor_desc(ptx::smem_u32(sm + Lay::oV), BN, 0);
      auto issue_s = [&](int j) {  // S_j = Q K_j^T
        const int s = j % NS;
        wait(&full[s], (j / NS) & 1);
        ptx::tc_fence_after();
        const uint32_t so = static_cast<uint32_t>(s * Lay::kKV);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tS, tc::desc_add(dQ, tc::kmajor_off(BM, kk)), tc::desc_add(dK, so + tc::kmajor_off(BN, kk)), idS,
                      kk > 0 ? 1u : 0u);
        ptx::mma_commit_e(s_full);
        if constexpr (Lay::SPLIT) ptx::mma_commit_e(k_empty);  // the K buffer may be refilled
      };
      wait(q_full, 0);
      issue_s(0);
      for (int j = 0; j < nkv; ++j) {
        if (j + 1 < nkv) {
          wait(s_consumed, j & 1);  // S_j is in the softmax registers: the S columns are free
          issue_s(j + 1);
        }
        wait(p_ready, j & 1);  // P_j written, O rescaled
        if constexpr (Lay::SPLIT) wait(v_full, j & 1);
        ptx::tc_fence_after();
        const uint32_t so = static_cast<uint32_t>((j % NS) * Lay::kKV);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          ptx::mma_ts_e(tO, tP + k * 8, tc::desc_add(dV, so + k * 16 * 128), idO, (j > 0 || k > 0) ? 1u : 0u);
        ptx::mma_commit_e(&empty[j % NS]);
        ptx::mma_commit_e(pv_done);
      }
      ptx::mma_commit_e(o_full);
    }
  } else if (Lay::SPLIT && warp == 6) {
    // ----------------------------------------------- V loader (d = 256)
    if (lane == 0 && ok) {
      for (int j = 0; j < nkv; ++j) {
        if (j >= 1) wait(&empty[0], (j - 1) & 1);  // P_{j-1} V_{j-1} has read the V buffer
        ptx::mbar_expect_tx(v_full, Lay::kKV);
        for (int c = 0; c < D / 64; ++c)
          ptx::tma_load_3d(sm + Lay::oV + c * BN * 128, &tmV, v_full, c * 64, (j0 + j) * BN, kvh);
      }
      if (nkv > 0) wait(&empty[0], (nkv - 1) & 1);
    }
  } else if constexpr (PB) {
    // ------------------------------- P^ b: thread r owns query row r, L is known
    const int r = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int64_t row = static_cast<int64_t>(rb) * BM + r;
    const float L2 = row < N ? lse_in[static_cast<int64_t>(bh) * N + row] * kLog2e : 0.f;
    const int lo_row = (WIN && causal) ? bd.row_lo(bh, row) : 0;
    const uint64_t c2 = tc::pk2f(scale_log2, scale_log2), nL2 = tc::pk2f(-L2, -L2);
    for (int j = 0; j < nkv; ++j) {
      wait(s_full, j & 1);
      ptx::tc_fence_after();
      const int kb = j0 + j;
      // Keys of this block past the row (causal), or past N, or below the row's window.
      const bool diag = causal ? (BN == BM ? kb == rb : kb * BN + BN - 1 > rb * BM) : (j == nkv - 1 && (N % BN) != 0);
      const bool low = WIN && causal && kb * BN < lo_last;
      const int klim = causal ? ((WIN || BN != BM) ? rb * BM + r - kb * BN : r) : N - 1 - kb * BN;
      const int klo = (WIN && causal) ? lo_row - kb * BN : 0;
      uint32_t v[BN / 32][32];
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) ptx::tmem_ld32(tS + lane_off + ch * 32, v[ch]);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(s_consumed);
      uint32_t pk[BN / 32][16];
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) {
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const float2 arg = tc::unpk2(tc::fma2(tc::pk2(v[ch][t], v[ch][t + 1]), c2, nL2));
          float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
          if (diag || low) {
            if (ch * 32 + t > klim || ch * 32 + t < klo) p0 = 0.f;
            if (ch * 32 + t + 1 > klim || ch * 32 + t + 1 < klo) p1 = 0.f;
          }
          pk[ch][t >> 1] = ptx::pack_bf16(p0, p1);
        }
      }
      if (j > 0) wait(pv_done, (j - 1) & 1);
      ptx::tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) ptx::tmem_st16(tP + lane_off + ch * 16, pk[ch]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(p_ready);
    }
    wait(o_full, 0);
    ptx::tc_fence_after();
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t v[32];
      ptx::tmem_ld32(tO + lane_off + ch * 32, v);
      ptx::tmem_wait_ld();
      if (row < N) {
        float4* dst = reinterpret_cast<float4*>(pb + (static_cast<int64_t>(bh) * N + row) * D + ch * 32);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          dst[u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                               __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
      }
    }
  } else {
    // ---------------------------------------- softmax: thread r owns query row r
    const int r = threadIdx.x;                       // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int64_t row = static_cast<int64_t>(rb) * BM + r;
    const int lo_row = (WIN && causal) ? bd.row_lo(bh, row) : 0;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nkv; ++j) {
      wait(s_full, j & 1);
      ptx::tc_fence_after();
      // Causal: only the diagonal block holds keys after some rows, and only the first
      // blocks keys below a row's window.  Otherwise only the last block can hold keys
      // past N (TMA reads them as zeros).
      const int kb = j0 + j;
      const bool diag = causal ? (BN == BM ? kb == rb : kb * BN + BN - 1 > rb * BM) : (j == nkv - 1 && (N % BN) != 0);
      const bool low = WIN && causal && kb * BN < lo_last;
      const int klim = causal ? ((WIN || BN != BM) ? rb * BM + r - kb * BN : r) : N - 1 - kb * BN;  // last visible
      const int klo = (WIN && causal) ? lo_row - kb * BN : 0;  // first visible key, relative
      // The whole BN-column S row in registers: BN / 32 loads, one wait.
      uint32_t v[BN / 32][32];
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) ptx::tmem_ld32(tS + lane_off + ch * 32, v[ch]);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(s_consumed);  // the MMA warp may now compute S_{j+1} into these columns
      if (diag || low) {
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch)
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (ch * 32 + t > klim || ch * 32 + t < klo) v[ch][t] = __float_as_uint(-INFINITY);
      }
      // Row max over 8 independent partial maxima (short dependency chains).
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch)
#pragma unroll
        for (int t = 0; t < 32; ++t) mx8[t & 7] = fmaxf(mx8[t & 7], __uint_as_float(v[ch][t]));
#pragma unroll
      for (int u = 1; u < 8; ++u) mx8[0] = fmaxf(mx8[0], mx8[u]);
      const float m_new = fmaxf(m, mx8[0]);
      const bool moved = (j > 0) && (m_new > m);
      const float alpha = moved ? ptx::ex2((m - m_new) * scale_log2) : 1.f;
      l *= alpha;
      m = m_new;
      // p = 2^((s - m) s log2 e): subtract first, then scale (masked entries are -inf -> 0).
      // Packed f32x2: (s - m) then * s log2 e for two keys per instruction.  A row with
      // no visible key yet (its window starts in a later block) subtracts 0, not -inf.
      const float msub = (WIN && m == -INFINITY) ? 0.f : m;
      const uint64_t nm2 = tc::pk2f(-msub, -msub), c2 = tc::pk2f(scale_log2, scale_log2);
      uint64_t rs4[4] = {0, 0, 0, 0};
      uint32_t pk[BN / 32][16];  // P_j as bf16 pairs, written once P_{j-1} V_{j-1} is done
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) {
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const float2 arg = tc::unpk2(tc::mul2(tc::add2(tc::pk2(v[ch][t], v[ch][t + 1]), nm2), c2));
          const float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
          const uint64_t P2 = tc::pk2f(p0, p1);
          rs4[(t >> 1) & 3] = tc::add2(rs4[(t >> 1) & 3], P2);
          pk[ch][t >> 1] = ptx::pack_bf16(p0, p1);
        }
      }
      if (j > 0) wait(pv_done, (j - 1) & 1);  // P_{j-1} V_{j-1} has read the P columns and updated O
      ptx::tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) ptx::tmem_st16(tP + lane_off + ch * 16, pk[ch]);  // keys ch*32 .. ch*32+31
      const float2 rsa = tc::unpk2(tc::add2(tc::add2(rs4[0], rs4[1]), tc::add2(rs4[2], rs4[3])));
      const float rs = rsa.x + rsa.y;
      if (__any_sync(0xffffffffu, moved)) {  // rescale O for rows whose max moved
        // up to 64 columns per round trip: both loads in flight, one wait, packed multiplies
        constexpr int R = D < 64 ? D / 32 : 2;
        const uint64_t a2 = tc::pk2f(alpha, alpha);
#pragma unroll
        for (int c0 = 0; c0 < D / 32; c0 += R) {
          uint32_t o[R][32];
#pragma unroll
          for (int u = 0; u < R; ++u) ptx::tmem_ld32(tO + lane_off + (c0 + u) * 32, o[u]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < R; ++u) {
#pragma unroll
            for (int t = 0; t < 32; t += 2) {
              const float2 v = tc::unpk2(tc::mul2(tc::pk2(o[u][t], o[u][t + 1]), a2));
              o[u][t] = __float_as_uint(v.x);
              o[u][t + 1] = __float_as_uint(v.y);
            }
            ptx::tmem_st32(tO + lane_off + (c0 + u) * 32, o[u]);
          }
        }
      }
      ptx::tmem_wait_st();
      l += rs;
      ptx::tc_fence_before();
      ptx::mbar_arrive(p_ready);
    }
    // ------------------------------------------------------------------ epilogue
    wait(o_full, 0);
    ptx::tc_fence_after();
    const float inv = 1.f / l;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t v[32];
      ptx::tmem_ld32(tO + lane_off + ch * 32, v);
      ptx::tmem_wait_ld();
      if (row < N && ch * 32 < dv) {  // columns past the head dim dv are padding
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2)
          pk[t >> 1] = ptx::pack_bf16(__uint_as_float(v[t]) * inv, __uint_as_float(v[t + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(O + (static_cast<int64_t>(bh) * N + row) * dv + ch * 32);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = make_uint4(pk[u * 4], pk[u * 4 + 1], pk[u * 4 + 2], pk[u * 4 + 3]);
      }
    }
    if (row < N) lse[static_cast<int64_t>(bh) * N + row] = m * scale + logf(l);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <int D, bool PB>
cudaError_t launch(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse,
                   const float* lse_in, float* pb, cudaStream_t st) {
  alignas(64) CUtensorMap mq, mk, mv;
  // Tensor maps over the true head dim p.d (<= D): TMA zero-fills columns p.d .. D-1,
  // which add nothing to any product.
  constexpr int BN = Layout<D>::BN;
  if (!make_tmap_bf16(&mq, Q, p.N, p.d, p.BH, BM) || !make_tmap_bf16(&mk, K, p.N, p.d, p.BHkv, BN) ||
      !make_tmap_bf16(&mv, V, p.N, p.d, p.BHkv, BN))
    return cudaErrorInvalidValue;
  const int nrb = static_cast<int>((p.N + BM - 1) / BM);
  const size_t smem = Layout<D>::bytes;
  auto kern = banded(p) ? fwd_kernel<D, PB, true> : fwd_kernel<D, PB, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(nrb * p.BH), Layout<D>::kThreads, smem, st>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(O), lse, lse_in, pb, static_cast<int>(p.N), nrb,
      static_cast<int>(p.BH), p.scale, p.scale * kLog2e, p.causal, make_band(p, eff_window_tc(p), false), p.group,
      static_cast<int>(p.d));
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_fwd(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse,
                   cudaStream_t st) {
  // d = 32 runs the d = 64 kernel and d = 96 the d = 128 one, zero-padded in shared memory.
  // d = 256: one K and one V buffer, each reloaded on its own (the Q tile alone takes 64 KB).
  return p.d <= 64    ? launch<64, false>(p, Q, K, V, O, lse, nullptr, nullptr, st)
         : p.d <= 128 ? launch<128, false>(p, Q, K, V, O, lse, nullptr, nullptr, st)
                      : launch<256, false>(p, Q, K, V, O, lse, nullptr, nullptr, st);
}

cudaError_t tc_bob_pb(const Problem& p, const void* Q, const void* K, const void* b, const float* lse, float* pb,
                      cudaStream_t st) {
  // Rows of bob_pb_cols(d) floats: 64 for d <= 64, 128 for d <= 128 (padding columns 0).
  return p.d <= 64 ? launch<64, true>(p, Q, K, b, nullptr, nullptr, lse, pb, st)
                   : launch<128, true>(p, Q, K, b, nullptr, nullptr, lse, pb, st);
}

uint32_t tc_fwd_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
