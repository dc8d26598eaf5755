// bf16 backward-over-backward (FlashBoB) on sm_103a, d = 64: a row pass and a
// column pass, every output block written once, nothing N x N in HBM.
//
// "FlashBoB: second-order attention", "Two scalar states replace quadratic
// tensors".  With a = gdQ, b = gdK, c = gdV, G = s(a K^T + Q b^T), H = dO c^T,
// dS = P * (dP - D), W = G * dS + P * H, the two per-row scalar states are
//   E_i = sum_j P_ij G_ij   and   F_i = F'_i - E_i D_i,  F'_i = sum_j W_ij.
// Row pass (CTA holds 128 query rows; 64-key blocks j <= i stream past):
//   tiles   [Q b^T | S] = Q [b_j; K_j]^T,  G += a K_j^T,  [H | dP] = dO [c_j; V_j]^T
//   outputs [X | U] += P [c_j | K_j],  X += (P G) V_j,  [Y | Z] += dS [b_j | K_j],
//           Y += W K_j   (128-wide products wherever two share an A operand)
//   end     gdO = X - E O,  gQ = s (Y - E Z - F' U); row states (L log2 e, E, D, F')
// (the corrections after the finished row are linear in E and F', so they are
// applied once per row: "partial sums accumulated early, corrected after").
// Column pass (CTA holds 128 keys; 64-query blocks i >= j stream past, with the
// row states re-read): transposed tiles, lanes = keys,
//   tiles   [S^T | K a^T] = K [Q_i; a_i]^T,  G^T += b Q_i^T,  dP^T = V dO_i^T,
//           H^T = c dO_i^T
//   dPbar = P (G - E),  Sbar = P (G (dP - D) - E dP + H - F) = P ((G - E)(dP - D) + H - F')
//   outputs gV += dPbar^T dO_i,  gK += dS^T a_i + Sbar^T Q_i;  end gK *= s.
// The row pass's tile products read both operands from 128-byte-swizzled shared
// memory (TMA); the column pass's take the held K, b, V, c from TMEM.  The output
// products take the bf16 tiles (P, P G, dS, W in the row pass; dPbar, dS, Sbar in
// the column pass) from TMEM as the A operand and the streamed block, MN-major,
// from shared memory as B.
//
// Rounding: the output products see bf16 copies P^, (PG)^, dS^, W^ of the tiles.
// The corrections use E_i = sum_j (PG)_ij (fp32) and a second state taken from
// those same copies,  F'_i = (sum_j W^_ij - E_i sum_j dS^_ij) / sum_j P^_ij,
// so that the row of Sbar the products effectively see, W^ - E dS^ - F' P^, sums
// to exactly zero (as the exact Sbar does) whatever the rounding of E.  In exact arithmetic these are the
// definitions above (sum dS = 0, sum P = 1); in bf16 they keep the rounding of W
// from being multiplied by the mean key, the same mechanism GProj removes from dQ
// ("FlashAttention bf16 gradient and GProj", "How the zero sum turns into a false
// gradient").  The stored state F'_i = sum_j W_ij uses the fp32 sums.
//
// Shift: every output is unchanged when a per-row constant g0_i is added to the row
// of G (dPbar and Sbar hold G only through G - E, and E moves with it).  A large
// mean of b (or of K) puts such a constant, s q_i.mean(b), into G, and the bf16
// copies (PG)^ and W^ would round it before E removes it.  The row pass therefore
// works with G - g0, g0_i = G at the first key of its first key block: (PG)^, W^, E and F'
// are those of the shifted G (F' = sum_j W_ij is shift-free since sum_j dS_ij = 0),
// and the stored E is shifted back for the column pass, which forms G - E in fp32.
//
// Row-pass TMEM: one 128-column tile region holding first [G | S] and then
// [H | dP] of the same key block, the four bf16 operands (32 columns each, the A
// operand of the output products), X, U, Y, Z 64 each = 512.  Column-pass TMEM:
// tile region 128, held K, b, V, c 128, operands 96, gV, gK 128.  An MMA with both
// operands in shared memory
// needs 8 KB per 128 x 128 x 16 step, which is the whole shared-memory bandwidth
// of the SM (128 B per clock); taking the output products' A operand from TMEM
// keeps the passes off that limit.  In both passes the compute warps copy tiles
// into registers and release their columns at once, so the next tile MMAs overlap
// the CUDA-core work; no TMEM region is read by one MMA while a later MMA with a
// different accumulator writes it (such MMAs carry no ordering guarantee).
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fbd {
namespace {

__device__ unsigned int g_err = 0;

constexpr int D = 64;
constexpr int BM = 128;
constexpr int BN = 64;
constexpr int kCompute = 256;
constexpr int kThreads = kCompute + 96;  // compute warps, TMA warp, tile-MMA warp, output-MMA warp
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTile = BN * D * 2;  // 8 KB: one streamed 64-row tile
constexpr int kHeld = BM * D * 2;  // 16 KB: one held 128-row tile

using tc::bf16_hi;
using tc::bf16_lo;
using tc::f;

// ================================================================ row pass
// Two MMA warps share the tensor pipe.  Per 64-key block j the tile warp issues
// [G | S](j) into the tile region once the compute warps have copied [H | dP](j-1)
// out (barrier `consumed_b`), then [H | dP](j) once they have copied [G | S](j)
// out (`consumed_a`); the output warp issues outputs(j) once the bf16 operands of
// block j are in TMEM (`ready`).  With one issuing warp the barrier waits between
// the phases left the pipe idle; with two, each warp's waits overlap the other's
// MMAs.  The compute warps turn S and G into P and PG while [H | dP] is computed.
// The operand columns are rewritten only after outputs(j-1) finished reading them
// (`out_done`); a stage is refilled once both warps have committed its MMAs.
struct RowLay {
  static constexpr int NS = 5;
  static constexpr int oQ = 0, odO = kHeld, oA = 2 * kHeld;
  static constexpr int oStage = 3 * kHeld;
  // One stage: c_j, V_j, b_j, K_j (8 KB each).  [c_j; V_j] and [b_j; K_j] are the
  // 128-row B operands of the tile products; K_j sits at a fixed positive offset
  // from c_j and from b_j, so [c_j | K_j] and [b_j | K_j] are 128-wide MN-major B
  // operands of the output products (two 64-column slabs, leading offset = gap).
  static constexpr int kStage = 4 * kTile;
  static constexpr int oc = 0, oV = kTile, ob = 2 * kTile, oKs = 3 * kTile;
  static constexpr int oRed = oStage + NS * kStage;
  static constexpr int oBar = oRed + 13 * BM * 4;
  static constexpr int bytes = oBar + 256;
  // TMEM: tile region [G | S] (Q b^T + a K^T, then Q K^T), later [H | dP] of the same
  // block; bf16 operands P^, (PG)^, dS^, W^; accumulators [X | U], [Y | Z].
  static constexpr int cG = 0, cS = 64, cH = 0, cdP = 64;
  static constexpr int cP = 128, cPG = 160, cdS = 192, cW = 224;
  static constexpr int cX = 256, cU = 320, cY = 384, cZ = 448;
};

// PAD: head dim hd < D (zero-padded in shared memory).  The unpadded instance sees
// the constant D, so its code is that of a kernel without the option.
// GP: GProj on the rounded dS of gQ's dS b product (the pre-pass left P^ b in `pb`);
// the coefficient rho_i goes to `rho_ws` for the column pass.
// WIN: a banded causal mask is in force (bd: the sliding window and/or the document
// bounds); the other instances carry none of it.
template <bool PAD, bool GP, bool WIN = false>
__global__ void __launch_bounds__(kThreads, 1)
    bob_row_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __nv_bfloat16* __restrict__ O,
                   const __nv_bfloat16* __restrict__ dO, const float* __restrict__ lse,
                   __nv_bfloat16* __restrict__ gQ, __nv_bfloat16* __restrict__ gdO, float4* __restrict__ ws,
                   const float* __restrict__ pb, float* __restrict__ rho_ws, int N, int Np, int nrb, int BH,
                   float scale, float c, int causal, Band bd, int G, int hd_arg) {
  const int hd = PAD ? hd_arg : D;
  using Lay = RowLay;
  constexpr int NS = Lay::NS;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* q_full = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
  uint64_t* full = q_full + 1;
  uint64_t* empty = full + NS;
  uint64_t* sa_full = empty + NS;     // [G | S] of the current block in TMEM
  uint64_t* sb_full = sa_full + 1;    // [H | dP] of the current block in TMEM
  uint64_t* consumed_a = sb_full + 1;
  uint64_t* consumed_b = consumed_a + 1;
  uint64_t* ready = consumed_b + 1;
  uint64_t* out_done = ready + 1;
  uint64_t* acc_full = out_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(sm + Lay::oRed);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Order ord = tc::grid_order(BH, nrb);
  const int bh = ord.bh;
  const int kvh = bh / G;          // the slice of K, V, b, c this query slice reads
  const int rb = nrb - 1 - ord.k;  // heaviest row blocks first (within a group of slices)
  // 64-key blocks this row block sees: up to its last row, or all of them when not causal
  const int j0 = (WIN && causal) ? bd.row_lo(bh, rb * BM) / BN : 0;  // first key block a row sees (banded mask bd)
  const int lo_last = (WIN && causal) ? bd.row_lo(bh, min(rb * BM + BM - 1, N - 1)) : 0;
  const int nkv = (causal ? ((rb + 1) * BM + BN - 1) / BN : (N + BN - 1) / BN) - j0;  // blocks j0 + j, j < nkv

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 2);  // released by the tile warp and by the output warp
    }
    ptx::mbar_init(sa_full, 1);
    ptx::mbar_init(sb_full, 1);
    ptx::mbar_init(consumed_a, kCompute);
    ptx::mbar_init(consumed_b, kCompute);
    ptx::mbar_init(ready, kCompute);
    ptx::mbar_init(out_done, 1);
    ptx::mbar_init(acc_full, 1);
    *abort_flag = (ptx::smem_u32(sm) & 1023u) ? 1 : 0;
    if (*abort_flag) atomicOr(&g_err, FBD_ERR_TIMEOUT);
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::BoundedWait wait{abort_flag, &g_err};
  const bool ok = *abort_flag == 0;

  if (warp == 8) {
    if (lane == 0 && ok) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmB);
      ptx::prefetch_tmap(&tmC);
      ptx::mbar_expect_tx(q_full, 3 * kHeld);
      ptx::tma_load_3d(sm + Lay::oQ, &tmQ, q_full, 0, rb * BM, bh);
      ptx::tma_load_3d(sm + Lay::odO, &tmdO, q_full, 0, rb * BM, bh);
      ptx::tma_load_3d(sm + Lay::oA, &tmA, q_full, 0, rb * BM, bh);
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS;
        if (j >= NS) wait(&empty[s], ((j / NS) - 1) & 1);
        uint8_t* st = sm + Lay::oStage + s * Lay::kStage;
        ptx::mbar_expect_tx(&full[s], 4 * kTile);
        ptx::tma_load_3d(st + Lay::oc, &tmC, &full[s], 0, (j0 + j) * BN, kvh);
        ptx::tma_load_3d(st + Lay::oV, &tmV, &full[s], 0, (j0 + j) * BN, kvh);
        ptx::tma_load_3d(st + Lay::ob, &tmB, &full[s], 0, (j0 + j) * BN, kvh);
        ptx::tma_load_3d(st + Lay::oKs, &tmK, &full[s], 0, (j0 + j) * BN, kvh);
      }
      for (int j = (nkv > NS ? nkv - NS : 0); j < nkv; ++j) wait(&empty[j % NS], (j / NS) & 1);
    }
  } else if (warp == 9) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t id128 = ptx::idesc_bf16(BM, 2 * BN, 0, 0);
      constexpr uint32_t id64 = ptx::idesc_bf16(BM, BN, 0, 0);
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage);
      // Descriptors at K-step 0 of stage 0.  A K-step moves a K-major operand by 32 B
      // and an MN-major one by 16 rows (2 KB); stage s adds s * kStage.
      const uint64_t dQ = tc::kmajor_desc(ptx::smem_u32(sm + Lay::oQ), BM, 0);
      const uint64_t ddO = tc::kmajor_desc(ptx::smem_u32(sm + Lay::odO), BM, 0);
      const uint64_t dA = tc::kmajor_desc(ptx::smem_u32(sm + Lay::oA), BM, 0);
      const uint64_t dBK = tc::kmajor_desc(sSt + Lay::ob, 2 * BN, 0);   // [b_j; K_j], K-major
      const uint64_t dKk = tc::kmajor_desc(sSt + Lay::oKs, BN, 0);      // K_j, K-major
      const uint64_t dCV = tc::kmajor_desc(sSt + Lay::oc, 2 * BN, 0);   // [c_j; V_j], K-major
      const uint32_t tG = tmem + Lay::cG, tH = tmem + Lay::cH;
      wait(q_full, 0);
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(&full[s], (j / NS) & 1);
        if (j > 0) wait(consumed_b, (j - 1) & 1);  // [H | dP] of block j-1 copied out of TMEM
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tG, tc::desc_add(dQ, 32 * kk), tc::desc_add(dBK, so + 32 * kk), id128, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tG, tc::desc_add(dA, 32 * kk), tc::desc_add(dKk, so + 32 * kk), id64, 1u);
        ptx::mma_commit_e(sa_full);
        wait(consumed_a, j & 1);  // [G | S] of block j copied out of TMEM
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tH, tc::desc_add(ddO, 32 * kk), tc::desc_add(dCV, so + 32 * kk), id128, kk > 0);
        ptx::mma_commit_e(sb_full);
        ptx::mma_commit_e(&empty[s]);
      }
    }
  } else if (warp == 10) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idO = ptx::idesc_bf16(BM, D, 0, 1);
      constexpr uint32_t idO2 = ptx::idesc_bf16(BM, 2 * D, 0, 1);
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage);
      const uint64_t dCK = ptx::sdesc_sw128(sSt + Lay::oc, Lay::oKs - Lay::oc, 1024);  // [c_j | K_j], MN-major
      const uint64_t dVm = tc::mnmajor_desc(sSt + Lay::oV, BN, 0);      // V_j, MN-major
      const uint64_t dBKm = ptx::sdesc_sw128(sSt + Lay::ob, Lay::oKs - Lay::ob, 1024);  // [b_j | K_j], MN-major
      const uint64_t dKm = tc::mnmajor_desc(sSt + Lay::oKs, BN, 0);     // K_j, MN-major
      const uint32_t tX = tmem + Lay::cX, tY = tmem + Lay::cY;
      const uint32_t tP = tmem + Lay::cP, tPG = tmem + Lay::cPG, tdS = tmem + Lay::cdS, tW = tmem + Lay::cW;
      for (int j = 0; j < nkv; ++j) {  // X, Y, Z, U += block j's operands x its streamed tiles
        const int s = j % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(ready, j & 1);
        wait(&full[s], (j / NS) & 1);  // already complete: the stage cannot refill before this warp releases it
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint32_t acc = (j > 0 || k > 0) ? 1u : 0u;
          const uint32_t kb = so + 2048 * k;
          // [X | U] += P [c | K],  X += (PG) V,  [Y | Z] += dS [b | K],  Y += W K
          ptx::mma_ts_e(tX, tP + 8 * k, tc::desc_add(dCK, kb), idO2, acc);
          ptx::mma_ts_e(tX, tPG + 8 * k, tc::desc_add(dVm, kb), idO, 1u);
          ptx::mma_ts_e(tY, tdS + 8 * k, tc::desc_add(dBKm, kb), idO2, acc);
          ptx::mma_ts_e(tY, tW + 8 * k, tc::desc_add(dKm, kb), idO, 1u);
        }
        ptx::mma_commit_e(&empty[s]);
        ptx::mma_commit_e(out_done);
      }
      ptx::mma_commit_e(acc_full);
    }
  } else {
    const int qd = warp & 3, hf = warp >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>(qd * 32) << 16;
    const int64_t row = static_cast<int64_t>(rb) * BM + r;
    const bool live = row < N;
    const int lo_row = (WIN && causal) ? bd.row_lo(bh, row) : 0;
    const size_t rowoff = (static_cast<size_t>(bh) * N + row) * hd;  // rows of hd <= D columns
    float part = 0.f;
    if (live && hf * 32 < hd) {  // columns past hd are padding
      const uint4* po = reinterpret_cast<const uint4*>(O + rowoff + hf * 32);
      const uint4* pg = reinterpret_cast<const uint4*>(dO + rowoff + hf * 32);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 o = po[u], g = pg[u];
        const uint32_t aw[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) part += bf16_lo(aw[e]) * bf16_lo(gw[e]) + bf16_hi(aw[e]) * bf16_hi(gw[e]);
      }
    }
    red[hf * BM + r] = part;
    tc::named_sync(1, kCompute);
    const float Dr = red[r] + red[BM + r];
    const float L2 = live ? lse[static_cast<size_t>(bh) * N + row] * kLog2e : 0.f;
    // Per-row sums as fp32 pairs (two keys per f32x2 instruction).
    uint64_t accE = 0, accF = 0;
    // Sums of the bf16 operands (even and odd keys apart), for the consistent-rounding state.
    float accW0 = 0.f, accW1 = 0.f, accdS0 = 0.f, accdS1 = 0.f, accP0 = 0.f, accP1 = 0.f;
    const uint64_t c2 = tc::pk2f(c, c), s2 = tc::pk2f(scale, scale);
    const uint64_t nL2 = tc::pk2f(-L2, -L2), nD2 = tc::pk2f(-Dr, -Dr);
    // The row's shift g0 lives in shared memory (red) and is read where it is used, so it
    // holds no register through the block's [H | dP] phase, where the registers run out.
    volatile float* g0p = red + 12 * BM + r;
    const int c0 = hf * 32;
    const uint32_t tOp = tmem + static_cast<uint32_t>(hf * 16) + lo;  // this thread's keys in the operand columns
    for (int j = 0; j < nkv; ++j) {
      wait(sa_full, j & 1);
      ptx::tc_fence_after();
      uint32_t sv[32], gv[32];
      ptx::tmem_ld32(tmem + Lay::cS + c0 + lo, sv);
      ptx::tmem_ld32(tmem + Lay::cG + c0 + lo, gv);
      if (j > 0) {  // block j-1's operand stores complete while this block's tiles load
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ready);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(consumed_a);  // the MMA warp may now write [H | dP] into the tile region
      if (j == 0) {  // the row's shift g0 = G at the first key of the first block (any key serves)
        if (hf == 0) red[12 * BM + r] = scale * f(gv[0]);
        tc::named_sync(1, kCompute);
      }
      const int kb = j0 + j;
      const int krel = kb * BN + c0 - rb * BM;
      // last visible key of this row, relative to the thread's first key of the block
      const int klim = causal ? r - krel : N - 1 - (kb * BN + c0);
      const int klo = (WIN && causal) ? lo_row - (kb * BN + c0) : 0;  // first visible key of the row, relative to column 0
      uint64_t P2[16], G2[16];
      uint32_t pP[16], pG[16], pS[16], pW[16];
      // P, PG from the [G | S] tiles (while [H | dP] is being computed)
      auto first = [&](auto masked) {
        const float g0 = *g0p;
        const uint64_t ng0 = tc::pk2f(-g0, -g0);
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const float2 arg = tc::unpk2(tc::fma2(tc::pk2(sv[t], sv[t + 1]), c2, nL2));
          float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
          if constexpr (decltype(masked)::value) {
            if (t > klim || t < klo) p0 = 0.f;
            if (t + 1 > klim || t + 1 < klo) p1 = 0.f;
          }
          const int idx = t >> 1;
          P2[idx] = tc::pk2f(p0, p1);
          G2[idx] = tc::fma2(tc::pk2(gv[t], gv[t + 1]), s2, ng0);  // G - g0
          const uint64_t pg2 = tc::mul2(P2[idx], G2[idx]);
          accE = tc::add2(accE, pg2);
          const float2 pg = tc::unpk2(pg2);
          pP[idx] = ptx::pack_bf16(p0, p1);
          pG[idx] = ptx::pack_bf16(pg.x, pg.y);
          accP0 = tc::add_bf16_lo(accP0, pP[idx]);
          accP1 = tc::add_bf16_hi(accP1, pP[idx]);
        }
      };
      // Causal: a block reaching past the first row of this CTA.  Otherwise: a block reaching past N.
      if (causal ? (krel + 31 > 0 || (WIN && kb * BN + c0 < lo_last)) : kb * BN + c0 + 32 > N)
        first(std::true_type{});
      else
        first(std::false_type{});
      wait(sb_full, j & 1);
      ptx::tc_fence_after();
      uint32_t dv[32], hv[32];
      ptx::tmem_ld32(tmem + Lay::cdP + c0 + lo, dv);
      ptx::tmem_ld32(tmem + Lay::cH + c0 + lo, hv);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(consumed_b);  // the MMA warp may now write the next block's [G | S]
      // dS, W from the [H | dP] tiles
#pragma unroll
      for (int t = 0; t < 32; t += 2) {
        const int idx = t >> 1;
        const uint64_t ds2 = tc::mul2(P2[idx], tc::add2(tc::pk2(dv[t], dv[t + 1]), nD2));
        const uint64_t w2 = tc::fma2(G2[idx], ds2, tc::mul2(P2[idx], tc::pk2(hv[t], hv[t + 1])));
        accF = tc::add2(accF, w2);
        const float2 ds = tc::unpk2(ds2), w = tc::unpk2(w2);
        pS[idx] = ptx::pack_bf16(ds.x, ds.y);
        pW[idx] = ptx::pack_bf16(w.x, w.y);
        accW0 = tc::add_bf16_lo(accW0, pW[idx]);
        accW1 = tc::add_bf16_hi(accW1, pW[idx]);
        accdS0 = tc::add_bf16_lo(accdS0, pS[idx]);
        accdS1 = tc::add_bf16_hi(accdS1, pS[idx]);
      }
      if (j > 0) wait(out_done, (j - 1) & 1);  // block j-1's products have read the operand columns
      ptx::tmem_st16(tOp + Lay::cP, pP);
      ptx::tmem_st16(tOp + Lay::cPG, pG);
      ptx::tmem_st16(tOp + Lay::cdS, pS);
      ptx::tmem_st16(tOp + Lay::cW, pW);  // completed (and `ready` arrived) at the next block's loads
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    ptx::mbar_arrive(ready);  // the last block's operands
    auto hsum = [](uint64_t x) {
      const float2 v = tc::unpk2(x);
      return v.x + v.y;
    };
    red[2 * BM + hf * BM + r] = hsum(accE);
    red[4 * BM + hf * BM + r] = hsum(accF);
    red[6 * BM + hf * BM + r] = accW0 + accW1;
    red[8 * BM + hf * BM + r] = accdS0 + accdS1;
    red[10 * BM + hf * BM + r] = accP0 + accP1;
    tc::named_sync(1, kCompute);
    const float E = red[2 * BM + r] + red[3 * BM + r];
    const float Fp = red[4 * BM + r] + red[5 * BM + r];
    const float sW = red[6 * BM + r] + red[7 * BM + r];
    const float sdS = red[8 * BM + r] + red[9 * BM + r];
    const float sP = red[10 * BM + r] + red[11 * BM + r];
    const float Fq = (sW - E * sdS) / sP;  // F' as seen through the bf16 operands
    wait(acc_full, 0);
    ptx::tc_fence_after();
    uint32_t xv[32], yv[32], zv[32], uv[32];
    ptx::tmem_ld32(tmem + Lay::cX + c0 + lo, xv);
    ptx::tmem_ld32(tmem + Lay::cY + c0 + lo, yv);
    ptx::tmem_ld32(tmem + Lay::cZ + c0 + lo, zv);
    ptx::tmem_ld32(tmem + Lay::cU + c0 + lo, uv);
    ptx::tmem_wait_ld();
    if (live && c0 < hd) {
      uint32_t ow[16];  // this thread's half of the O row (32 bf16), read again here
      const uint4* po = reinterpret_cast<const uint4*>(O + rowoff + c0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 o = po[u];
        ow[4 * u] = o.x;
        ow[4 * u + 1] = o.y;
        ow[4 * u + 2] = o.z;
        ow[4 * u + 3] = o.w;
      }
      uint32_t go[16], gq[16];
#pragma unroll
      for (int t = 0; t < 32; t += 2) {
        const float o0 = bf16_lo(ow[t >> 1]), o1 = bf16_hi(ow[t >> 1]);
        go[t >> 1] = ptx::pack_bf16(f(xv[t]) - E * o0, f(xv[t + 1]) - E * o1);
      }
      uint4* d0 = reinterpret_cast<uint4*>(gdO + rowoff + c0);
#pragma unroll
      for (int u = 0; u < 4; ++u) d0[u] = make_uint4(go[4 * u], go[4 * u + 1], go[4 * u + 2], go[4 * u + 3]);
      if constexpr (GP) {  // Y holds dS^ b: subtract rho_i (P^ b)_i, rho_i = sum_j dS^_ij / sum_j P^_ij
        const float rho = sdS / sP;
        const float4* pp = reinterpret_cast<const float4*>(pb + (static_cast<size_t>(bh) * N + row) * D + c0);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 q = pp[u];
          const float qv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) yv[4 * u + e] = __float_as_uint(fmaf(-rho, qv[e], f(yv[4 * u + e])));
        }
      }
#pragma unroll
      for (int t = 0; t < 32; t += 2)
        gq[t >> 1] = ptx::pack_bf16(scale * (f(yv[t]) - E * f(zv[t]) - Fq * f(uv[t])),
                                    scale * (f(yv[t + 1]) - E * f(zv[t + 1]) - Fq * f(uv[t + 1])));
      uint4* d1 = reinterpret_cast<uint4*>(gQ + rowoff + c0);
#pragma unroll
      for (int u = 0; u < 4; ++u) d1[u] = make_uint4(gq[4 * u], gq[4 * u + 1], gq[4 * u + 2], gq[4 * u + 3]);
    }
    if (hf == 0 && row < Np) {  // row states, negated, pair-interleaved (see the column pass)
      // F' = F + E D = sum_j W_ij is what the column pass needs (its (G - E)(dP - D) form).
      // The row past N of an odd-length slice gets zeros, so the column pass never reads
      // unwritten workspace (its P is masked to 0 there).
      float* wf = reinterpret_cast<float*>(ws) + static_cast<size_t>(bh) * Np * 4;
      const int64_t k2 = row & ~static_cast<int64_t>(1);
      const int odd = static_cast<int>(row & 1);
      wf[k2 * 4 + odd] = live ? -L2 : 0.f;
      wf[k2 * 4 + 2 + odd] = live ? -(E + *g0p) : 0.f;  // the unshifted E
      wf[(k2 + 1) * 4 + odd] = live ? -Dr : 0.f;
      wf[(k2 + 1) * 4 + 2 + odd] = live ? -Fp : 0.f;
    }
    if constexpr (GP) {  // -rho_i, one float per row (rows up to the pitch written, as zeros past N)
      const int64_t pitch = bob_rho_pitch(N);
      if (hf == 0 && row < pitch) rho_ws[static_cast<size_t>(bh) * pitch + row] = live ? -(sdS / sP) : 0.f;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}


// ============================================================= column pass
// Same hand-off as the row pass: the tile region holds first [S^T | G^T] and then
// [dP^T | H^T] of the same 64-query block (barriers `consumed_a`, `consumed_b`), a
// tile warp and an output warp issue the MMAs, `out_done` guards the operand
// columns.  The held key-side operands K, b, V, c sit in TMEM as the A operands of
// the tile products, so those MMAs read only the streamed operand from shared
// memory; with both operands in shared memory they took the SM's whole
// shared-memory bandwidth and starved the compute warps' reads of the row states.
// Per element the compute warps form
//   P = 2^(S c - L log2 e),  dPbar = P (G - E),  dS = P (dP - D),
//   Sbar = P ((G - E)(dP - D) + H - F')          (F' = F + E D, stored by the row pass)
// GP (GProj): the stage also holds the 64 queries' coefficients -rho (256 bytes behind
// the states); the compute warps write bf16(-rho_i P_ij) into TMEM (cPT) and the output
// warp adds that operand times a_i to gK, the key term of the projection.
template <bool GP>
struct ColLayT {
  static constexpr int NS = 8;
  static constexpr int kStat = BN * 16;
  static constexpr int kRho = BN * 4;
  static constexpr int kStage = 3 * kTile + 2048;  // [Q_i; a_i], dO_i, row states (+ GProj coefficients)
  static constexpr int oStage = 0;
  static constexpr int oBar = oStage + NS * kStage;
  static constexpr int bytes = oBar + 256;
  // TMEM: tile region, held bf16 A operands K, b, V, c (32 columns each), the bf16
  // output operands dPbar, dS, Sbar (32 each), accumulators gV, gK; with GP P^ (32).
  static constexpr int cT = 0, cK = 128, cB = 160, cV = 192, cC = 224, cOp = 256, cgV = 352, cgK = 416, cPT = 480;
};
static_assert(ColLayT<true>::bytes <= 232448, "column pass shared memory");

// The column pass runs 16 compute warps (warp w: TMEM lanes 32 (w % 4) .., queries
// 16 (w / 4) .. of each 64-query block), then the TMA, tile-MMA and output-MMA warps.
constexpr int kColCompute = 512;
constexpr int kColThreads = kColCompute + 96;
constexpr int wTma = kColCompute / 32, wTile = wTma + 1, wOut = wTma + 2;
// GR: grouped key/value heads (G > 1).  The G == 1 instance keeps the plain tile loop.
// PAD as in the row pass.  GP as in ColLayT (tmRho: the coefficients, laid out as the states).
template <bool GR, bool PAD, bool GP, bool WIN = false>
__global__ void __launch_bounds__(kColThreads, 1)
    bob_col_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmdO, const __grid_constant__ CUtensorMap tmSt,
                   const __grid_constant__ CUtensorMap tmRho, const __nv_bfloat16* __restrict__ Kp, const __nv_bfloat16* __restrict__ Bp,
                   const __nv_bfloat16* __restrict__ Vp, const __nv_bfloat16* __restrict__ Cp,
                   __nv_bfloat16* __restrict__ gK, __nv_bfloat16* __restrict__ gV, int N, int BHkv, float scale,
                   float c, int causal, Band bd, int G, int hd_arg) {
  const int hd = PAD ? hd_arg : D;
  using Lay = ColLayT<GP>;
  constexpr int NS = Lay::NS;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
  uint64_t* empty = full + NS;
  uint64_t* held_ready = empty + NS;  // K, b, V, c of this key block in TMEM
  uint64_t* sa_full = held_ready + 1;
  uint64_t* sb_full = sa_full + 1;
  uint64_t* consumed_a = sb_full + 1;
  uint64_t* consumed_b = consumed_a + 1;
  uint64_t* ready = consumed_b + 1;
  uint64_t* out_done = ready + 1;
  uint64_t* acc_full = out_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + BM - 1) / BM;
  const tc::Order ord = tc::grid_order(BHkv, nkb);
  const int kvh = ord.bh;  // key/value slice; its G query slices are kvh * G + h, h < G
  const int kb = ord.k;  // first key blocks have the most rows: first
  const int nq = (N + BN - 1) / BN;
  const int i0 = causal ? (kb * BM) / BN : 0;  // first query block that sees this key block
  // query blocks per query slice: up to the last query any key of the block sees (bd.key_hi)
  const int ntile = ((WIN && causal) ? bd.key_hi(kvh, min(kb * BM + BM - 1, N - 1)) / BN + 1 : nq) - i0;
  const int hi_first = (WIN && causal) ? bd.key_hi(kvh, kb * BM) : 0;  // the block's first key's last query
  const int nt = GR ? G * ntile : ntile;       // tiles t = h * ntile + (i - i0), one gK, gV

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 2);  // released by the tile warp and by the output warp
    }
    ptx::mbar_init(held_ready, kColCompute);
    ptx::mbar_init(sa_full, 1);
    ptx::mbar_init(sb_full, 1);
    ptx::mbar_init(consumed_a, kColCompute);
    ptx::mbar_init(consumed_b, kColCompute);
    ptx::mbar_init(ready, kColCompute);
    ptx::mbar_init(out_done, 1);
    ptx::mbar_init(acc_full, 1);
    *abort_flag = (ptx::smem_u32(sm) & 1023u) ? 1 : 0;
    if (*abort_flag) atomicOr(&g_err, FBD_ERR_TIMEOUT);
    ptx::fence_mbar_init();
  }
  if (warp == wTile) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::BoundedWait wait{abort_flag, &g_err};
  const bool ok = *abort_flag == 0;

  if (warp == wTma) {
    if (lane == 0 && ok) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmdO);
      ptx::prefetch_tmap(&tmSt);
      if constexpr (GP) ptx::prefetch_tmap(&tmRho);
      for (int t = 0; t < nt; ++t) {
        const int h = GR ? t / ntile : 0, s = t % NS, i = i0 + t - h * ntile, bh = GR ? kvh * G + h : kvh;
        if (t >= NS) wait(&empty[s], ((t / NS) - 1) & 1);
        uint8_t* st = sm + Lay::oStage + s * Lay::kStage;
        ptx::mbar_expect_tx(&full[s], 3 * kTile + Lay::kStat + (GP ? Lay::kRho : 0));
        ptx::tma_load_3d(st, &tmQ, &full[s], 0, i * BN, bh);
        ptx::tma_load_3d(st + kTile, &tmA, &full[s], 0, i * BN, bh);
        ptx::tma_load_3d(st + 2 * kTile, &tmdO, &full[s], 0, i * BN, bh);
        ptx::tma_load_3d(st + 3 * kTile, &tmSt, &full[s], 0, i * BN, bh);
        if constexpr (GP) ptx::tma_load_3d(st + 3 * kTile + Lay::kStat, &tmRho, &full[s], 0, i * (BN / 4), bh);
      }
      for (int t = (nt > NS ? nt - NS : 0); t < nt; ++t) wait(&empty[t % NS], (t / NS) & 1);
    }
  } else if (warp == wTile) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t id128 = ptx::idesc_bf16(BM, 2 * BN, 0, 0);
      constexpr uint32_t id64 = ptx::idesc_bf16(BM, BN, 0, 0);
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage);
      // B descriptors at K-step 0 of stage 0 (a K-step adds 32 B, stage s adds s * kStage).
      const uint64_t dQA = tc::kmajor_desc(sSt, 2 * BN, 0);            // [Q_i; a_i], K-major
      const uint64_t dQk = tc::kmajor_desc(sSt, BN, 0);                // Q_i, K-major
      const uint64_t ddOk = tc::kmajor_desc(sSt + 2 * kTile, BN, 0);   // dO_i, K-major
      const uint32_t tT = tmem + Lay::cT, tK = tmem + Lay::cK, tB = tmem + Lay::cB;
      const uint32_t tV = tmem + Lay::cV, tC = tmem + Lay::cC;
      wait(held_ready, 0);
      for (int t = 0; t < nt; ++t) {
        const int s = t % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(&full[s], (t / NS) & 1);
        if (t > 0) wait(consumed_b, (t - 1) & 1);  // [dP^T | H^T] of block t-1 copied out of TMEM
        ptx::tc_fence_after();
        // [S^T | K a^T] = K [Q_i; a_i]^T,  G^T += b Q_i^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ts_e(tT, tK + 8 * kk, tc::desc_add(dQA, so + 32 * kk), id128, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ts_e(tT + BN, tB + 8 * kk, tc::desc_add(dQk, so + 32 * kk), id64, 1u);
        ptx::mma_commit_e(sa_full);
        wait(consumed_a, t & 1);  // [S^T | G^T] of block t copied out of TMEM
        ptx::tc_fence_after();
        // dP^T = V dO_i^T,  H^T = c dO_i^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ts_e(tT, tV + 8 * kk, tc::desc_add(ddOk, so + 32 * kk), id64, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ts_e(tT + BN, tC + 8 * kk, tc::desc_add(ddOk, so + 32 * kk), id64, kk > 0);
        ptx::mma_commit_e(sb_full);
        ptx::mma_commit_e(&empty[s]);
      }
    }
  } else if (warp == wOut) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idO = ptx::idesc_bf16(BM, D, 0, 1);
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage);
      const uint64_t dQm = tc::mnmajor_desc(sSt, BN, 0);               // Q_i, MN-major
      const uint64_t dAm = tc::mnmajor_desc(sSt + kTile, BN, 0);       // a_i, MN-major
      const uint64_t ddOm = tc::mnmajor_desc(sSt + 2 * kTile, BN, 0);  // dO_i, MN-major
      const uint32_t tOp = tmem + Lay::cOp, tgV = tmem + Lay::cgV, tgK = tmem + Lay::cgK;
      const uint32_t tPT = tmem + Lay::cPT;
      for (int t = 0; t < nt; ++t) {
        const int s = t % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(ready, t & 1);
        wait(&full[s], (t / NS) & 1);  // already complete: the stage cannot refill before this warp releases it
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint32_t acc = (t > 0 || k > 0) ? 1u : 0u;
          const uint32_t kb2 = so + 2048 * k;
          // gV += dPbar^T dO_i,  gK += dS^T a_i + Sbar^T Q_i
          ptx::mma_ts_e(tgV, tOp + k * 8, tc::desc_add(ddOm, kb2), idO, acc);
          ptx::mma_ts_e(tgK, tOp + 32 + k * 8, tc::desc_add(dAm, kb2), idO, acc);
          ptx::mma_ts_e(tgK, tOp + 64 + k * 8, tc::desc_add(dQm, kb2), idO, 1u);
          if constexpr (GP) ptx::mma_ts_e(tgK, tPT + k * 8, tc::desc_add(dAm, kb2), idO, 1u);  // (-rho P)^T a_i
        }
        ptx::mma_commit_e(&empty[s]);
        ptx::mma_commit_e(out_done);
      }
      ptx::mma_commit_e(acc_full);
    }
  } else {
    const int qd = warp & 3, hf = warp >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>(qd * 32) << 16;
    const int key = kb * BM + r;
    const int c0 = hf * 16;  // this thread's 16 queries of each block (and 16 of the head dim)
    const int khi = (WIN && causal) ? bd.key_hi(kvh, key) : 0;  // the last query this key is seen by
    {  // K, b, V, c rows of this key, elements 16 hf .. 16 hf + 15, into TMEM (A operands)
      const __nv_bfloat16* src[4] = {Kp, Bp, Vp, Cp};
      const uint32_t col[4] = {Lay::cK, Lay::cB, Lay::cV, Lay::cC};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t w[8];
        if (key < N && c0 < hd) {
          const uint4* g = reinterpret_cast<const uint4*>(src[m] + (static_cast<size_t>(kvh) * N + key) * hd + c0);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint4 v = g[u];
            w[4 * u] = v.x;
            w[4 * u + 1] = v.y;
            w[4 * u + 2] = v.z;
            w[4 * u + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) w[u] = 0u;
        }
        ptx::tmem_st8(tmem + col[m] + static_cast<uint32_t>(hf * 8) + lo, w);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(held_ready);
    }
    const uint64_t c2 = tc::pk2f(c, c), s2 = tc::pk2f(scale, scale);
    const uint32_t tOpT = tmem + Lay::cOp + static_cast<uint32_t>(hf * 8) + lo;
    for (int t = 0; t < nt; ++t) {
      const int s = t % NS, i = GR ? i0 + t % ntile : i0 + t;
      // Row states of the 64 queries, pair-interleaved: float4 2m = (-L2, -L2', -E, -E'),
      // float4 2m+1 = (-D, -D', -F', -F'') of queries 2m, 2m+1 of the block.
      const float4* stat =
          reinterpret_cast<const float4*>(sm + Lay::oStage + s * Lay::kStage + 3 * kTile) + c0;
      const int qbase = i * BN + c0;
      wait(sa_full, t & 1);
      ptx::tc_fence_after();
      uint32_t sv[16], gv[16];
      ptx::tmem_ld16(tmem + Lay::cT + c0 + lo, sv);
      ptx::tmem_ld16(tmem + Lay::cT + BN + c0 + lo, gv);
      if (t > 0) {  // block t-1's operand stores complete while this block's tiles load
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ready);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(consumed_a);  // the tile warp may now write [dP^T | H^T]
      uint64_t P2[8], GE2[8];
      uint32_t pDP[8], pDS[8], pSB[8], pPT[GP ? 8 : 1];
      // GP: -rho of this thread's 16 queries (the stage's coefficient tile)
      const float4* nrho = reinterpret_cast<const float4*>(sm + Lay::oStage + s * Lay::kStage + 3 * kTile +
                                                           Lay::kStat) + c0 / 4;
      auto first = [&](auto masked) {  // P and P (G - E) from [S^T | G^T]
#pragma unroll
        for (int u = 0; u < 16; u += 2) {
          const float4 A = stat[u];
          const float2 arg = tc::unpk2(tc::fma2(tc::pk2(sv[u], sv[u + 1]), c2, tc::pk2f(A.x, A.y)));
          float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
          if constexpr (decltype(masked)::value) {
            const int q0 = qbase + u;
            if ((causal && (q0 < key || (WIN && q0 > khi))) || q0 >= N) p0 = 0.f;
            if ((causal && (q0 + 1 < key || (WIN && q0 + 1 > khi))) || q0 + 1 >= N) p1 = 0.f;
          }
          const int idx = u >> 1;
          P2[idx] = tc::pk2f(p0, p1);
          GE2[idx] = tc::fma2(tc::pk2(gv[u], gv[u + 1]), s2, tc::pk2f(A.z, A.w));  // G - E
          const float2 vdp = tc::unpk2(tc::mul2(P2[idx], GE2[idx]));
          pDP[idx] = ptx::pack_bf16(vdp.x, vdp.y);
        }
      };
      // Causal mask only in the first blocks (queries before this CTA's last key) and in
      // those past the window of its first key; past N only in the last block.
      if ((causal && (qbase < kb * BM + BM || (WIN && qbase + 15 > hi_first))) || qbase + 16 > N)
        first(std::true_type{});
      else
        first(std::false_type{});
      wait(sb_full, t & 1);
      ptx::tc_fence_after();
      uint32_t dv[16], hv[16];
      ptx::tmem_ld16(tmem + Lay::cT + c0 + lo, dv);
      ptx::tmem_ld16(tmem + Lay::cT + BN + c0 + lo, hv);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(consumed_b);  // the tile warp may now write the next block's [S^T | G^T]
#pragma unroll
      for (int u = 0; u < 16; u += 2) {  // dS and Sbar from [dP^T | H^T]
        const float4 Bs = stat[u + 1];
        const int idx = u >> 1;
        const uint64_t dmd = tc::add2(tc::pk2(dv[u], dv[u + 1]), tc::pk2f(Bs.x, Bs.y));  // dP - D
        const float2 vds = tc::unpk2(tc::mul2(P2[idx], dmd));
        const uint64_t in = tc::add2(tc::fma2(GE2[idx], dmd, tc::pk2(hv[u], hv[u + 1])), tc::pk2f(Bs.z, Bs.w));
        const float2 vsb = tc::unpk2(tc::mul2(P2[idx], in));
        pDS[idx] = ptx::pack_bf16(vds.x, vds.y);
        pSB[idx] = ptx::pack_bf16(vsb.x, vsb.y);
      }
      if constexpr (GP) {  // bf16(-rho_i P_ij), formed once dP and H are out of the registers
#pragma unroll
        for (int u = 0; u < 16; u += 4) {
          const float4 r4 = nrho[u >> 2];
          const float2 a0 = tc::unpk2(tc::mul2(P2[u >> 1], tc::pk2f(r4.x, r4.y)));
          const float2 a1 = tc::unpk2(tc::mul2(P2[(u >> 1) + 1], tc::pk2f(r4.z, r4.w)));
          pPT[u >> 1] = ptx::pack_bf16(a0.x, a0.y);
          pPT[(u >> 1) + 1] = ptx::pack_bf16(a1.x, a1.y);
        }
      }
      if (t > 0) wait(out_done, (t - 1) & 1);  // block t-1's products have read the operand columns
      if constexpr (GP) ptx::tmem_st8(tmem + Lay::cPT + static_cast<uint32_t>(hf * 8) + lo, pPT);
      ptx::tmem_st8(tOpT, pDP);
      ptx::tmem_st8(tOpT + 32, pDS);
      ptx::tmem_st8(tOpT + 64, pSB);  // completed (and `ready` arrived) at the next block's loads
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    ptx::mbar_arrive(ready);  // the last block's operands
    wait(acc_full, 0);
    ptx::tc_fence_after();
    uint32_t av[16], bv[16];
    ptx::tmem_ld16(tmem + Lay::cgV + c0 + lo, av);
    ptx::tmem_ld16(tmem + Lay::cgK + c0 + lo, bv);
    ptx::tmem_wait_ld();
    if (key < N && c0 < hd) {
      const size_t rowoff = (static_cast<size_t>(kvh) * N + key) * hd;
      uint32_t ov[8], ok2[8];
#pragma unroll
      for (int u = 0; u < 16; u += 2) {
        ov[u >> 1] = ptx::pack_bf16(f(av[u]), f(av[u + 1]));
        ok2[u >> 1] = ptx::pack_bf16(scale * f(bv[u]), scale * f(bv[u + 1]));
      }
      uint4* dvp = reinterpret_cast<uint4*>(gV + rowoff + c0);
      uint4* dkp = reinterpret_cast<uint4*>(gK + rowoff + c0);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        dvp[u] = make_uint4(ov[4 * u], ov[4 * u + 1], ov[4 * u + 2], ov[4 * u + 3]);
        dkp[u] = make_uint4(ok2[4 * u], ok2[4 * u + 1], ok2[4 * u + 2], ok2[4 * u + 3]);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == wTile) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t tc_bob(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* lse, const void* a, const void* b, const void* cc, void* gQ, void* gK, void* gV,
                   void* gdO, bool gproj, float4* ws, int passes, cudaStream_t st) {
  if (p.d > D) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap q128, do128, a128, k64, v64, b64, c64;
  alignas(64) CUtensorMap q64, a64, do64, s64, r64;
  // GProj: the coefficients follow the states, P^ b follows them (see internal.h).
  float4* rho = gproj ? bob_rho_region(ws, p) : ws;
  float* pbuf = gproj ? bob_pb_region(ws, p) : nullptr;
  const int64_t N = p.N, BH = p.BH, Np = (p.N + 1) & ~static_cast<int64_t>(1), d = p.d;
  // Tensor maps over the true head dim d <= D: TMA zero-fills the padding columns.
  if (!make_tmap_bf16(&q128, Q, N, d, BH, BM) || !make_tmap_bf16(&do128, dO, N, d, BH, BM) ||
      !make_tmap_bf16(&a128, a, N, d, BH, BM) || !make_tmap_bf16(&k64, K, N, d, p.BHkv, BN) ||
      !make_tmap_bf16(&v64, V, N, d, p.BHkv, BN) || !make_tmap_bf16(&b64, b, N, d, p.BHkv, BN) ||
      !make_tmap_bf16(&c64, cc, N, d, p.BHkv, BN) || !make_tmap_bf16(&q64, Q, N, d, BH, BN) ||
      !make_tmap_bf16(&a64, a, N, d, BH, BN) || !make_tmap_bf16(&do64, dO, N, d, BH, BN) ||
      !make_tmap_stats(&s64, ws, Np, BH, BN) ||
      !make_tmap_stats(&r64, rho, bob_rho_pitch(N) / 4, BH, BN / 4))  // 64 floats = 16 float4 rows
    return cudaErrorInvalidValue;
  const float c = p.scale * kLog2e;
  const int nrb = static_cast<int>((N + BM - 1) / BM);
  cudaError_t e = cudaSuccess;
  // The GProj instances take the general forms (runtime head dim, grouped tile loop),
  // which also serve d = 64 and ungrouped heads.
  if (passes & 1) {
    if (gproj && (e = tc_bob_pb(p, Q, K, b, lse, pbuf, st)) != cudaSuccess) return e;
    // Windowed: the general forms (runtime head dim, grouped tile loop in the column pass).
    auto row = banded(p) ? (gproj ? bob_row_kernel<true, true, true> : bob_row_kernel<true, false, true>)
               : gproj ? bob_row_kernel<true, true> : d < D ? bob_row_kernel<true, false> : bob_row_kernel<false, false>;
    e = cudaFuncSetAttribute(row, cudaFuncAttributeMaxDynamicSharedMemorySize, RowLay::bytes);
    if (e != cudaSuccess) return e;
    row<<<static_cast<unsigned>(nrb * BH), kThreads, RowLay::bytes, st>>>(
        q128, do128, a128, k64, v64, b64, c64, static_cast<const __nv_bfloat16*>(O),
        static_cast<const __nv_bfloat16*>(dO), lse, static_cast<__nv_bfloat16*>(gQ),
        static_cast<__nv_bfloat16*>(gdO), ws, pbuf, reinterpret_cast<float*>(rho), static_cast<int>(N),
        static_cast<int>(Np), nrb, static_cast<int>(BH), p.scale, c, p.causal, make_band(p, eff_window_tc(p), false),
        p.group, static_cast<int>(d));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (!(passes & 2)) return cudaSuccess;
  auto col = banded(p) ? (gproj ? bob_col_kernel<true, true, true, true> : bob_col_kernel<true, true, false, true>)
             : gproj ? bob_col_kernel<true, true, true>
             : p.group > 1 ? (d < D ? bob_col_kernel<true, true, false> : bob_col_kernel<true, false, false>)
                           : (d < D ? bob_col_kernel<false, true, false> : bob_col_kernel<false, false, false>);
  const int cbytes = gproj ? ColLayT<true>::bytes : ColLayT<false>::bytes;
  e = cudaFuncSetAttribute(col, cudaFuncAttributeMaxDynamicSharedMemorySize, cbytes);
  if (e != cudaSuccess) return e;
  col<<<static_cast<unsigned>(nrb * p.BHkv), kColThreads, cbytes, st>>>(
      q64, a64, do64, s64, r64, static_cast<const __nv_bfloat16*>(K), static_cast<const __nv_bfloat16*>(b),
      static_cast<const __nv_bfloat16*>(V), static_cast<const __nv_bfloat16*>(cc), static_cast<__nv_bfloat16*>(gK),
      static_cast<__nv_bfloat16*>(gV), static_cast<int>(N), static_cast<int>(p.BHkv), p.scale, c, p.causal,
      make_band(p, eff_window_tc(p), true), p.group, static_cast<int>(d));
  return cudaGetLastError();
}

uint32_t tc_bob_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
