// bf16 causal attention backward without GProj, with 128-wide score tiles: the row
// pass (dQ) at d = 64 and d = 128 (96 zero-padded), the column pass (dK, dV) at
// d = 64 (at d = 128 its tiles and accumulators would need 640 TMEM columns; the
// 64-wide column pass of tc_bwd.cu, which reads the same row statistics, runs
// there).
//
// Same mathematics as tc_bwd.cu ("Flash attention for trading models",
// "Backward pass: recompute instead of store"): P = 2^(S s log2 e - L log2 e),
// dP = dO V^T, dS = P (dP - D); dQ = s dS K, dK = s dS^T Q, dV = P^T dO, each
// output block written once.  What differs is the shape of the work: both the
// held and the streamed blocks are 128 rows, so every score-tile MMA is
// M = N = 128 (a 64-wide MMA takes about 70 % longer per flop on this GPU), and
// the tiles live in TMEM single-buffered, released early:
//   - the compute warps copy their slice of the S and dP tiles into registers and
//     arrive on `consumed`; the MMA warp may then compute the next block's tiles
//     into the same columns while the CUDA cores work on this block;
//   - the bf16 operands (dS, and P in the column pass) have their own TMEM
//     columns, rewritten only after the previous block's products have read them
//     (`out_done`).
// Warps 0-15 compute (warp w: TMEM lanes 32(w%4).., tile columns 32(w/4)..),
// warp 16 issues TMA loads, warp 17 allocates TMEM and issues the MMAs.
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fbd {
namespace {

__device__ unsigned int g_err = 0;

constexpr int D = 64;
constexpr int BW = 128;        // held and streamed block rows
constexpr int NS = 4;          // stages of streamed blocks
constexpr int kCW = 16;        // compute warps
constexpr int kCompute = kCW * 32;
constexpr int kThreads = kCompute + 96;  // + TMA warp, tile-MMA warp, output-MMA warp
constexpr int kC = 32;         // tile columns per compute thread (128 / 4 column groups)
constexpr int DG = D / 4;      // output columns per compute thread
constexpr int kTile = BW * D * 2;  // 16 KB
constexpr float kLog2e = 1.4426950408889634f;

using tc::bf16_hi;
using tc::bf16_lo;

// Shared boilerplate: barriers, TMEM allocation, bounded waits (NSX stages).
template <int NSX>
struct SyncT {
  static constexpr int NS = NSX;
  uint64_t* held_full;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* s_full;
  uint64_t* consumed;
  uint64_t* ready;
  uint64_t* out_done;
  uint64_t* acc_full;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  __device__ SyncT(uint8_t* base) {
    held_full = reinterpret_cast<uint64_t*>(base);
    full = held_full + 1;
    empty = full + NS;
    s_full = empty + NS;
    consumed = s_full + 1;
    ready = consumed + 1;
    out_done = ready + 1;
    acc_full = out_done + 1;
    tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  }
  __device__ void init(const uint8_t* sm) {
    ptx::mbar_init(held_full, 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 2);  // released by the tile warp and by the output warp
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(consumed, kCompute);
    ptx::mbar_init(ready, kCompute);
    ptx::mbar_init(out_done, 1);
    ptx::mbar_init(acc_full, 1);
    *abort_flag = (ptx::smem_u32(sm) & 1023u) ? 1 : 0;
    if (*abort_flag) atomicOr(&g_err, FBD_ERR_TIMEOUT);
    ptx::fence_mbar_init();
  }
};
using Sync = SyncT<NS>;

// ================================================================ row pass
// DR = 64, or 128 (d = 96, 128: the held Q, dO and two 64-column slabs per tile, two
// stages; TMEM S 128 + dP 128 + dS 64 + dQ 128 = 448 columns).
// GP (d = 64 only): GProj.  The bf16 P^ fed to a second output product P^ K (TMEM
// P^ 64 + PK 64 columns: 512 in all) and the row sums of dS^ and P^ give
// rho = sum dS^ / sum P^ and dQ = s (dS^ K - rho P^ K), the product of the projected
// row ("FlashAttention bf16 gradient and GProj", "How the zero sum turns into a
// false gradient"); -rho goes to the row statistics for the column pass.
template <int DR, bool GP = false>
struct RowLay {
  static_assert(!GP || DR == 64, "GProj rows at d = 64 only (TMEM)");
  static constexpr int NSR = DR == 64 ? NS : 2;
  static constexpr int kTileR = BW * DR * 2;
  static constexpr int DGR = DR / 4;  // dQ columns per compute thread
  static constexpr int oQ = 0, odO = kTileR, oK = 2 * kTileR, oV = oK + NSR * kTileR;
  static constexpr int oRed = oV + NSR * kTileR;  // float [4][BW]: D; with GProj [12][BW]: and the sums of dS^, P^
  static constexpr int oBar = oRed + (GP ? 12 : 4) * BW * 4;
  static constexpr int bytes = oBar + 256;
  static constexpr int cS = 0, cdP = 128, cdS = 256, cP = 320, cdQ = GP ? 384 : 320, cPK = cdQ + DR;
};
static_assert(RowLay<128>::bytes <= 232448, "row pass shared memory at d = 128");

// WIN: a banded causal mask is in force (bd: the sliding window and/or the document
// bounds); the other instances carry none of it.
template <int DR, bool GP, bool WIN = false>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_row_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
               const float* __restrict__ lse, __nv_bfloat16* __restrict__ dQ, float4* __restrict__ ws, int N, int Np,
               int nrb, int BH, float scale, float c, int causal, Band bd, int G, int dv) {
  using Lay = RowLay<DR, GP>;
  constexpr int NS = Lay::NSR, kTile = Lay::kTileR, DG = Lay::DGR, D = DR;
  extern __shared__ __align__(1024) uint8_t sm[];
  SyncT<NS> sy(sm + Lay::oBar);
  float* red = reinterpret_cast<float*>(sm + Lay::oRed);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Order ord = tc::grid_order(BH, nrb);
  const int bh = ord.bh;
  const int rb = nrb - 1 - ord.k;  // heaviest first within a group of slices
  // 128-key blocks j0 + j, j < nkv: up to rb (all blocks when not causal), from the first
  // block a row of this block sees under the banded mask bd (window and/or documents)
  const int j0 = (WIN && causal) ? bd.row_lo(bh, rb * BW) / BW : 0;
  const int lo_last = (WIN && causal) ? bd.row_lo(bh, min(rb * BW + BW - 1, N - 1)) : 0;
  const int nkv = (causal ? rb + 1 : nrb) - j0;

  if (threadIdx.x == 0) sy.init(sm);
  if (warp == kCW + 1) {
    ptx::tmem_alloc(sy.tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *sy.tmem_slot;
  const ptx::BoundedWait wait{sy.abort_flag, &g_err};
  const bool ok = *sy.abort_flag == 0;

  if (warp == kCW) {
    if (lane == 0 && ok) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::mbar_expect_tx(sy.held_full, 2 * kTile);
      for (int cc = 0; cc < D / 64; ++cc) {  // 64-column slabs, BW rows each
        ptx::tma_load_3d(sm + Lay::oQ + cc * BW * 128, &tmQ, sy.held_full, cc * 64, rb * BW, bh);
        ptx::tma_load_3d(sm + Lay::odO + cc * BW * 128, &tmdO, sy.held_full, cc * 64, rb * BW, bh);
      }
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS;
        if (j >= NS) wait(&sy.empty[s], ((j / NS) - 1) & 1);
        ptx::mbar_expect_tx(&sy.full[s], 2 * kTile);
        for (int cc = 0; cc < D / 64; ++cc) {
          ptx::tma_load_3d(sm + Lay::oK + s * kTile + cc * BW * 128, &tmK, &sy.full[s], cc * 64, (j0 + j) * BW,
                           bh / G);
          ptx::tma_load_3d(sm + Lay::oV + s * kTile + cc * BW * 128, &tmV, &sy.full[s], cc * 64, (j0 + j) * BW,
                           bh / G);
        }
      }
      for (int j = (nkv > NS ? nkv - NS : 0); j < nkv; ++j) wait(&sy.empty[j % NS], (j / NS) & 1);
    }
  } else if (warp == kCW + 1) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idS = ptx::idesc_bf16(BW, BW, 0, 0);
      // Descriptors at K-step 0 of stage 0, stepped with one add per MMA.
      const uint64_t dQ = tc::kmajor_desc(ptx::smem_u32(sm + Lay::oQ), BW, 0);
      const uint64_t ddO = tc::kmajor_desc(ptx::smem_u32(sm + Lay::odO), BW, 0);
      const uint32_t sK = ptx::smem_u32(sm + Lay::oK), sV = ptx::smem_u32(sm + Lay::oV);
      const uint64_t dKk = tc::kmajor_desc(sK, BW, 0), dVk = tc::kmajor_desc(sV, BW, 0);
      const uint32_t tS = tmem + Lay::cS, tdP = tmem + Lay::cdP;
      wait(sy.held_full, 0);
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS;
        wait(&sy.full[s], (j / NS) & 1);
        if (j > 0) wait(sy.consumed, (j - 1) & 1);  // tiles of block j-1 are in registers
        ptx::tc_fence_after();
        const uint32_t so = static_cast<uint32_t>(s * kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tS, tc::desc_add(dQ, tc::kmajor_off(BW, kk)), tc::desc_add(dKk, so + tc::kmajor_off(BW, kk)), idS,
                      kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tdP, tc::desc_add(ddO, tc::kmajor_off(BW, kk)), tc::desc_add(dVk, so + tc::kmajor_off(BW, kk)),
                      idS, kk > 0);
        ptx::mma_commit_e(sy.s_full);
        ptx::mma_commit_e(&sy.empty[s]);
      }
    }
  } else if (warp == kCW + 2) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idQ = ptx::idesc_bf16(BW, D, 0, 1);
      const uint64_t dKm = tc::mnmajor_desc(ptx::smem_u32(sm + Lay::oK), BW, 0);
      const uint32_t tdQ = tmem + Lay::cdQ, tdS = tmem + Lay::cdS, tP = tmem + Lay::cP, tPK = tmem + Lay::cPK;
      for (int t = 0; t < nkv; ++t) {  // dQ += dS_t K_t (PK += P_t K_t), then release the stage and the operands
        const int s = t % NS;
        wait(sy.ready, t & 1);
        wait(&sy.full[s], (t / NS) & 1);  // already complete: the stage cannot refill before this warp releases it
        ptx::tc_fence_after();
        const uint32_t so = static_cast<uint32_t>(s * kTile);
#pragma unroll
        for (int k = 0; k < BW / 16; ++k) {
          ptx::mma_ts_e(tdQ, tdS + k * 8, tc::desc_add(dKm, so + 2048 * k), idQ, (t > 0 || k > 0));
          if constexpr (GP) ptx::mma_ts_e(tPK, tP + k * 8, tc::desc_add(dKm, so + 2048 * k), idQ, (t > 0 || k > 0));
        }
        ptx::mma_commit_e(&sy.empty[s]);
        ptx::mma_commit_e(sy.out_done);
      }
      ptx::mma_commit_e(sy.acc_full);
    }
  } else {
    const int qd = warp & 3, cg = warp >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>(qd * 32) << 16;
    const int64_t row = static_cast<int64_t>(rb) * BW + r;
    const bool live = row < N;
    const size_t rowoff = (static_cast<size_t>(bh) * N + row) * dv;  // rows of dv <= D columns
    float part = 0.f;
    if (live) {  // this thread's quarter of D_r = dO_r . O_r (none in the padding)
      const uint4* po = reinterpret_cast<const uint4*>(O + rowoff + cg * DG);
      const uint4* pg = reinterpret_cast<const uint4*>(dO + rowoff + cg * DG);
#pragma unroll
      for (int u = 0; u < DG / 8; ++u) {
        if (cg * DG + 8 * u >= dv) break;
        const uint4 a = po[u], g = pg[u];
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) part += bf16_lo(aw[e]) * bf16_lo(gw[e]) + bf16_hi(aw[e]) * bf16_hi(gw[e]);
      }
    }
    red[cg * BW + r] = part;
    tc::named_sync(1, kCompute);
    const float Dr = red[r] + red[BW + r] + red[2 * BW + r] + red[3 * BW + r];
    const float L2 = live ? lse[static_cast<size_t>(bh) * N + row] * kLog2e : 0.f;
    const uint64_t c2 = tc::pk2f(c, c), nL2 = tc::pk2f(-L2, -L2), nD2 = tc::pk2f(-Dr, -Dr);
    const int c0 = cg * kC;
    const int lo_row = (WIN && causal) ? bd.row_lo(bh, row) : 0;
    uint64_t accR = 0, accP = 0;  // GProj: sums of the bf16 dS and P fed to the products
    for (int j = 0; j < nkv; ++j) {
      wait(sy.s_full, j & 1);
      ptx::tc_fence_after();
      uint32_t sv[kC], pv[kC];
      ptx::tmem_ld32(tmem + Lay::cS + c0 + lo, sv);
      ptx::tmem_ld32(tmem + Lay::cdP + c0 + lo, pv);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sy.consumed);
      uint32_t dsk[kC / 2], pkk[GP ? kC / 2 : 1];
      const int kb = j0 + j;
      const int klim = causal ? (WIN ? rb * BW + r - kb * BW : r) : N - 1 - kb * BW;  // last visible key, relative
      const int klo = (WIN && causal) ? lo_row - kb * BW : 0;  // first visible key, relative
      auto block = [&](auto masked) {
#pragma unroll
        for (int t = 0; t < kC; t += 2) {
          const float2 arg = tc::unpk2(tc::fma2(tc::pk2(sv[t], sv[t + 1]), c2, nL2));
          float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
          if constexpr (decltype(masked)::value) {
            // Causal: the diagonal block (keys past the row) and the blocks below a
            // row's window.  Otherwise the last block: keys at or past N.
            if (c0 + t > klim || c0 + t < klo) p0 = 0.f;
            if (c0 + t + 1 > klim || c0 + t + 1 < klo) p1 = 0.f;
          }
          const float2 ds = tc::unpk2(tc::mul2(tc::pk2f(p0, p1), tc::add2(tc::pk2(pv[t], pv[t + 1]), nD2)));
          dsk[t >> 1] = ptx::pack_bf16(ds.x, ds.y);
          if constexpr (GP) {
            pkk[t >> 1] = ptx::pack_bf16(p0, p1);
            accR = tc::add2(accR, tc::bf2_to_f2(dsk[t >> 1]));
            accP = tc::add2(accP, tc::bf2_to_f2(pkk[t >> 1]));
          }
        }
      };
      if (causal ? (kb == rb || (WIN && kb * BW < lo_last)) : (j == nkv - 1 && (N % BW) != 0))
        block(std::true_type{});
      else
        block(std::false_type{});
      if (j > 0) wait(sy.out_done, (j - 1) & 1);  // the previous block's dQ product has read dS
      ptx::tmem_st16(tmem + Lay::cdS + c0 / 2 + lo, dsk);
      if constexpr (GP) ptx::tmem_st16(tmem + Lay::cP + c0 / 2 + lo, pkk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sy.ready);
    }
    float rho = 0.f;
    if constexpr (GP) {  // rho_r = sum dS^ / sum P^ over the whole row (four column groups)
      const float2 vr = tc::unpk2(accR), vp = tc::unpk2(accP);
      red[4 * BW + cg * BW + r] = vr.x + vr.y;
      red[8 * BW + cg * BW + r] = vp.x + vp.y;
      tc::named_sync(1, kCompute);
      rho = (red[4 * BW + r] + red[5 * BW + r] + red[6 * BW + r] + red[7 * BW + r]) /
            (red[8 * BW + r] + red[9 * BW + r] + red[10 * BW + r] + red[11 * BW + r]);
    }
    wait(sy.acc_full, 0);
    ptx::tc_fence_after();
    uint32_t a[DG], pkv[GP ? DG : 1];
    if constexpr (DG == 16) {
      ptx::tmem_ld16(tmem + Lay::cdQ + cg * DG + lo, a);
      if constexpr (GP) ptx::tmem_ld16(tmem + Lay::cPK + cg * DG + lo, pkv);
    } else {
      ptx::tmem_ld32(tmem + Lay::cdQ + cg * DG + lo, a);
    }
    ptx::tmem_wait_ld();
    if constexpr (GP) {
#pragma unroll
      for (int t = 0; t < DG; ++t) a[t] = __float_as_uint(tc::f(a[t]) - rho * tc::f(pkv[t]));
    }
#pragma unroll
    for (int q = 0; q < DG / 16; ++q) {  // runs of 16 columns; none of them in the padding past dv
      if (live && cg * DG + q * 16 < dv) {
        uint32_t o[8];
#pragma unroll
        for (int t = 0; t < 16; t += 2)
          o[t >> 1] = ptx::pack_bf16(scale * tc::f(a[q * 16 + t]), scale * tc::f(a[q * 16 + t + 1]));
        uint4* dst = reinterpret_cast<uint4*>(dQ + rowoff + cg * DG + q * 16);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    if (cg == 0 && row < Np) {  // row statistics, negated, pair-interleaved (format shared with tc_bwd.cu)
      // The row past N of an odd-length slice gets zeros: the column pass reads it (with P = 0).
      float* wf = reinterpret_cast<float*>(ws) + static_cast<size_t>(bh) * Np * 4;
      const int64_t k2 = row & ~static_cast<int64_t>(1);
      const int odd = static_cast<int>(row & 1);
      wf[k2 * 4 + odd] = live ? -L2 : 0.f;
      wf[k2 * 4 + 2 + odd] = live ? -Dr : 0.f;
      wf[(k2 + 1) * 4 + odd] = live ? -rho : 0.f;
      wf[(k2 + 1) * 4 + 2 + odd] = 0.f;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kCW + 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ============================================================= column pass
// GP: GProj.  The key correction -sum_i rho_i P^_ij Q_i is a third output product
// that reuses the P^T operand: dK += P^T (-rho Q_i), with -rho_i Q_i (bf16) written by
// the compute warps into one more shared-memory tile in Q's layout, so the TMEM map
// stays that of the plain pass (a separate -rho P^ operand would need 576 columns).
template <bool GP = false>
struct ColLayT {
  static constexpr int kStat = BW * 16;
  static constexpr int kStage = 2 * kTile + kStat;  // Q_i, dO_i, statistics
  static constexpr int oK = 0, oV = kTile, oStage = 2 * kTile;
  static constexpr int oRQ = oStage + NS * kStage;  // GProj: -rho Q_i of the current block
  static constexpr int oBar = oRQ + (GP ? kTile : 0);
  static constexpr int bytes = oBar + 256;
  static constexpr int cS = 0, cdP = 128, cP = 256, cdS = 320, cdV = 384, cdK = 448;
};
using ColLay = ColLayT<false>;
static_assert(ColLayT<true>::bytes <= 232448 && ColLayT<true>::oRQ % 1024 == 0, "GProj column layout");

// GR: grouped key/value heads (G > 1).  The G == 1 instance keeps the plain tile loop.
template <bool GR, bool GP, bool WIN = false>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_col_wide_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
               const __grid_constant__ CUtensorMap tmSt, __nv_bfloat16* __restrict__ dK,
               __nv_bfloat16* __restrict__ dV, int N, int nb, int BHkv, float scale, float c, int causal, Band bd,
               int G, int dv) {
  using Lay = ColLayT<GP>;
  extern __shared__ __align__(1024) uint8_t sm[];
  Sync sy(sm + Lay::oBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Order ord = tc::grid_order(BHkv, nb);
  const int kvh = ord.bh;        // key/value slice; its G query slices are kvh * G + h, h < G
  const int kb = ord.k;          // first key blocks have the most query blocks: first
  const int i0 = causal ? kb : 0;  // first query block that sees this key block
  // query blocks per query slice: up to the last query any key of the block sees (the
  // banded mask bd: queries i <= bd.key_hi(key))
  const int ntile = ((WIN && causal) ? bd.key_hi(kvh, min(kb * BW + BW - 1, N - 1)) / BW + 1 : nb) - i0;
  const int hi_first = (WIN && causal) ? bd.key_hi(kvh, kb * BW) : 0;  // the block's first key's last query
  const int nt = GR ? G * ntile : ntile;  // tiles t = h * ntile + (i - i0), summed into one dK, dV

  if (threadIdx.x == 0) sy.init(sm);
  if (warp == kCW + 1) {
    ptx::tmem_alloc(sy.tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *sy.tmem_slot;
  const ptx::BoundedWait wait{sy.abort_flag, &g_err};
  const bool ok = *sy.abort_flag == 0;

  if (warp == kCW) {
    if (lane == 0 && ok) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmdO);
      ptx::prefetch_tmap(&tmSt);
      ptx::mbar_expect_tx(sy.held_full, 2 * kTile);
      ptx::tma_load_3d(sm + Lay::oK, &tmK, sy.held_full, 0, kb * BW, kvh);
      ptx::tma_load_3d(sm + Lay::oV, &tmV, sy.held_full, 0, kb * BW, kvh);
      for (int t = 0; t < nt; ++t) {
        const int h = GR ? t / ntile : 0, s = t % NS, i = i0 + t - h * ntile, bh = GR ? kvh * G + h : kvh;
        if (t >= NS) wait(&sy.empty[s], ((t / NS) - 1) & 1);
        uint8_t* st = sm + Lay::oStage + s * Lay::kStage;
        ptx::mbar_expect_tx(&sy.full[s], 2 * kTile + Lay::kStat);
        ptx::tma_load_3d(st, &tmQ, &sy.full[s], 0, i * BW, bh);
        ptx::tma_load_3d(st + kTile, &tmdO, &sy.full[s], 0, i * BW, bh);
        ptx::tma_load_3d(st + 2 * kTile, &tmSt, &sy.full[s], 0, i * BW, bh);
      }
      for (int t = (nt > NS ? nt - NS : 0); t < nt; ++t) wait(&sy.empty[t % NS], (t / NS) & 1);
    }
  } else if (warp == kCW + 1) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idS = ptx::idesc_bf16(BW, BW, 0, 0);
      // Descriptors at K-step 0 of stage 0, stepped with one add per MMA.
      const uint64_t dK = tc::kmajor_desc(ptx::smem_u32(sm + Lay::oK), BW, 0);
      const uint64_t dV = tc::kmajor_desc(ptx::smem_u32(sm + Lay::oV), BW, 0);
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage);
      const uint64_t dQk = tc::kmajor_desc(sSt, BW, 0), ddOk = tc::kmajor_desc(sSt + kTile, BW, 0);
      const uint32_t tS = tmem + Lay::cS, tdP = tmem + Lay::cdP;
      wait(sy.held_full, 0);
      for (int t = 0; t < nt; ++t) {
        const int s = t % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(&sy.full[s], (t / NS) & 1);
        if (t > 0) wait(sy.consumed, (t - 1) & 1);
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tS, tc::desc_add(dK, tc::kmajor_off(BW, kk)), tc::desc_add(dQk, so + tc::kmajor_off(BW, kk)), idS,
                      kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tdP, tc::desc_add(dV, tc::kmajor_off(BW, kk)), tc::desc_add(ddOk, so + tc::kmajor_off(BW, kk)),
                      idS, kk > 0);
        ptx::mma_commit_e(sy.s_full);
        ptx::mma_commit_e(&sy.empty[s]);
      }
    }
  } else if (warp == kCW + 2) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idKV = ptx::idesc_bf16(BW, D, 0, 1);
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage);
      const uint64_t dQm = tc::mnmajor_desc(sSt, BW, 0), ddOm = tc::mnmajor_desc(sSt + kTile, BW, 0);
      const uint32_t tP = tmem + Lay::cP, tdS = tmem + Lay::cdS, tdV = tmem + Lay::cdV, tdK = tmem + Lay::cdK;
      const uint64_t dRQm = tc::mnmajor_desc(ptx::smem_u32(sm + Lay::oRQ), BW, 0);  // GProj: -rho Q_i
      for (int t = 0; t < nt; ++t) {  // dV += P^T dO_i, dK += dS^T Q_i (+ P^T (-rho Q_i))
        const int s = t % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(sy.ready, t & 1);
        wait(&sy.full[s], (t / NS) & 1);  // already complete: the stage cannot refill before this warp releases it
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < BW / 16; ++k) {
          const uint32_t acc = (t > 0 || k > 0) ? 1u : 0u;
          ptx::mma_ts_e(tdV, tP + k * 8, tc::desc_add(ddOm, so + 2048 * k), idKV, acc);
          ptx::mma_ts_e(tdK, tdS + k * 8, tc::desc_add(dQm, so + 2048 * k), idKV, acc);
          if constexpr (GP) ptx::mma_ts_e(tdK, tP + k * 8, tc::desc_add(dRQm, 2048 * k), idKV, 1u);
        }
        ptx::mma_commit_e(&sy.empty[s]);
        ptx::mma_commit_e(sy.out_done);
      }
      ptx::mma_commit_e(sy.acc_full);
    }
  } else {
    const int qd = warp & 3, cg = warp >> 2;
    const int r = qd * 32 + lane;  // key row of the held block (TMEM lane) in the epilogue
    const uint32_t lo = static_cast<uint32_t>(qd * 32) << 16;
    const int key = kb * BW + r;
    const int c0 = cg * kC;
    // Score tiles are read with the 16-lane shapes, so that a thread sees 8 queries
    // of its 32 (pairs 2(t%4) + 8k, k < 4) for 4 keys (quarter rows t/4 + 8m, m < 4):
    // the row statistics of 4 query pairs stay in registers for the whole block.
    const int g4 = lane >> 2, q4 = lane & 3;
    // last query each of this thread's four keys (rows g4 + 16 h + 8 m of its quarter) sees
    int khi[2][2] = {{0, 0}, {0, 0}};
    if constexpr (WIN) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < 2; ++m) khi[h][m] = bd.key_hi(kvh, kb * BW + qd * 32 + g4 + 16 * h + 8 * m);
    }
    const uint64_t c2 = tc::pk2f(c, c);
    for (int t = 0; t < nt; ++t) {
      const int s = t % NS, i = GR ? i0 + t % ntile : i0 + t;
      wait(sy.s_full, t & 1);
      ptx::tc_fence_after();
      uint32_t sv[2][16], pv[2][16];  // [lanes +0 / +16 of the quarter][repetition k, (row, row+8) x (col, col+1)]
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t la = lo + (static_cast<uint32_t>(16 * h) << 16);
        ptx::tmem_ld16x256_x4(tmem + Lay::cS + c0 + la, sv[h]);
        ptx::tmem_ld16x256_x4(tmem + Lay::cdP + c0 + la, pv[h]);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sy.consumed);
      // Statistics of the block's queries, pair-interleaved and negated:
      // float4 2m = (-L2, -L2', -D, -D') of queries 2m, 2m+1.
      const float4* st = reinterpret_cast<const float4*>(sm + Lay::oStage + s * Lay::kStage + 2 * kTile) + c0;
      float4 A[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) A[k] = st[8 * k + 2 * q4];
      const int qbase = i * BW + c0 + 2 * q4;   // query of column (k = 0, col 0)
      const int kbase = kb * BW + qd * 32 + g4;  // key of (h = 0, row 0)
      uint32_t pk[2][8], dk[2][8];  // [h][2k + (row, row+8)]
      auto block = [&](auto masked) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const int e = 4 * k + 2 * m;
              const float2 arg =
                  tc::unpk2(tc::fma2(tc::pk2(sv[h][e], sv[h][e + 1]), c2, tc::pk2f(A[k].x, A[k].y)));
              float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
              if constexpr (decltype(masked)::value) {
                const int q0 = qbase + 8 * k, kk = kbase + 16 * h + 8 * m;
                if ((causal && (q0 < kk || (WIN && q0 > khi[h][m]))) || q0 >= N) p0 = 0.f;
                if ((causal && (q0 + 1 < kk || (WIN && q0 + 1 > khi[h][m]))) || q0 + 1 >= N) p1 = 0.f;
              }
              const float2 ds = tc::unpk2(
                  tc::mul2(tc::pk2f(p0, p1), tc::add2(tc::pk2(pv[h][e], pv[h][e + 1]), tc::pk2f(A[k].z, A[k].w))));
              pk[h][2 * k + m] = ptx::pack_bf16(p0, p1);
              dk[h][2 * k + m] = ptx::pack_bf16(ds.x, ds.y);
            }
      };
      // the diagonal block, a block reaching past the window of the block's first key, or past N
      if ((causal && (GR ? i == kb : t == 0)) || (WIN && causal && i * BW + BW - 1 > hi_first) ||
          i * BW + c0 + kC > N)
        block(std::true_type{});
      else
        block(std::false_type{});
      if (t > 0) wait(sy.out_done, (t - 1) & 1);  // the previous block's products have read P, dS (and -rho Q)
      if constexpr (GP) {
        // -rho_q Q_q of the block's 128 queries, 16 bytes (8 columns) per chunk, written at
        // the chunk's own offset (the 128-byte swizzle keeps a chunk within its row q).
        const uint8_t* qt = sm + Lay::oStage + s * Lay::kStage;
        const float* stf = reinterpret_cast<const float*>(qt + 2 * kTile);
#pragma unroll
        for (int m = 0; m < kTile / 16 / kCompute; ++m) {
          const int ch = static_cast<int>(threadIdx.x) + m * kCompute;
          const int q = ch >> 3;
          const float nrho = stf[((q >> 1) * 2 + 1) * 4 + (q & 1)];  // -rho of query q
          const uint4 v = reinterpret_cast<const uint4*>(qt)[ch];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = ptx::pack_bf16(nrho * bf16_lo(w[e]), nrho * bf16_hi(w[e]));
          reinterpret_cast<uint4*>(sm + Lay::oRQ)[ch] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        ptx::fence_proxy_async_smem();  // visible to the tensor core before `ready`
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t la = lo + (static_cast<uint32_t>(16 * h) << 16);
        ptx::tmem_st16x128_x4(tmem + Lay::cP + c0 / 2 + la, pk[h]);
        ptx::tmem_st16x128_x4(tmem + Lay::cdS + c0 / 2 + la, dk[h]);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sy.ready);
    }
    wait(sy.acc_full, 0);
    ptx::tc_fence_after();
    uint32_t a[DG], g[DG];
    ptx::tmem_ld16(tmem + Lay::cdV + cg * DG + lo, a);
    ptx::tmem_ld16(tmem + Lay::cdK + cg * DG + lo, g);
    ptx::tmem_wait_ld();
    if (key < N && cg * DG < dv) {
      const size_t rowoff = (static_cast<size_t>(kvh) * N + key) * dv;
      uint32_t ov[DG / 2], okk[DG / 2];
#pragma unroll
      for (int u = 0; u < DG; u += 2) {
        ov[u >> 1] = ptx::pack_bf16(tc::f(a[u]), tc::f(a[u + 1]));
        okk[u >> 1] = ptx::pack_bf16(scale * tc::f(g[u]), scale * tc::f(g[u + 1]));
      }
      uint4* dvp = reinterpret_cast<uint4*>(dV + rowoff + cg * DG);
      uint4* dk2 = reinterpret_cast<uint4*>(dK + rowoff + cg * DG);
      dvp[0] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
      dvp[1] = make_uint4(ov[4], ov[5], ov[6], ov[7]);
      dk2[0] = make_uint4(okk[0], okk[1], okk[2], okk[3]);
      dk2[1] = make_uint4(okk[4], okk[5], okk[6], okk[7]);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kCW + 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t tc_bwd_wide(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes,
                        cudaStream_t st, bool gproj) {
  // GProj: d <= 64 only (TMEM).
  if (gproj && p.d > 64) return cudaErrorInvalidValue;
  if (p.d > 64) {  // d = 96, 128: the row pass only (the column pass would need 640 TMEM columns)
    if (p.d > 128 || (passes & 2)) return cudaErrorInvalidValue;
    alignas(64) CUtensorMap q, g, k, v;
    const int64_t N = p.N, BH = p.BH, Np = (p.N + 1) & ~static_cast<int64_t>(1), d = p.d;
    if (!make_tmap_bf16(&q, Q, N, d, BH, BW) || !make_tmap_bf16(&g, dO, N, d, BH, BW) ||
        !make_tmap_bf16(&k, K, N, d, p.BHkv, BW) || !make_tmap_bf16(&v, V, N, d, p.BHkv, BW))
      return cudaErrorInvalidValue;
    const int nb = static_cast<int>((N + BW - 1) / BW);
    auto row = banded(p) ? bwd_row_wide_kernel<128, false, true> : bwd_row_wide_kernel<128, false, false>;
    cudaError_t e = cudaFuncSetAttribute(row, cudaFuncAttributeMaxDynamicSharedMemorySize, RowLay<128>::bytes);
    if (e != cudaSuccess) return e;
    row<<<static_cast<unsigned>(nb * BH), kThreads, RowLay<128>::bytes, st>>>(
        q, g, k, v, static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), lse,
        static_cast<__nv_bfloat16*>(dQ), ws, static_cast<int>(N), static_cast<int>(Np), nb, static_cast<int>(BH),
        p.scale, p.scale * kLog2e, p.causal, make_band(p, eff_window_tc(p), false), p.group, static_cast<int>(d));
    return cudaGetLastError();
  }
  alignas(64) CUtensorMap q, g, k, v, s;
  const int64_t N = p.N, BH = p.BH, Np = (p.N + 1) & ~static_cast<int64_t>(1), d = p.d;
  // Tensor maps over the true head dim d <= D: TMA zero-fills the padding columns.
  if (!make_tmap_bf16(&q, Q, N, d, BH, BW) || !make_tmap_bf16(&g, dO, N, d, BH, BW) ||
      !make_tmap_bf16(&k, K, N, d, p.BHkv, BW) || !make_tmap_bf16(&v, V, N, d, p.BHkv, BW) ||
      !make_tmap_stats(&s, ws, Np, BH, BW))
    return cudaErrorInvalidValue;
  const float c = p.scale * kLog2e;
  const int nb = static_cast<int>((N + BW - 1) / BW);
  cudaError_t e = cudaSuccess;
  if (passes & 1) {
    auto row = banded(p) ? (gproj ? bwd_row_wide_kernel<64, true, true> : bwd_row_wide_kernel<64, false, true>)
                            : (gproj ? bwd_row_wide_kernel<64, true> : bwd_row_wide_kernel<64, false>);
    const int bytes = gproj ? RowLay<64, true>::bytes : RowLay<64, false>::bytes;
    e = cudaFuncSetAttribute(row, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    row<<<static_cast<unsigned>(nb * BH), kThreads, bytes, st>>>(
        q, g, k, v, static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), lse,
        static_cast<__nv_bfloat16*>(dQ), ws, static_cast<int>(N), static_cast<int>(Np), nb, static_cast<int>(BH),
        p.scale, c, p.causal, make_band(p, eff_window_tc(p), false), p.group, static_cast<int>(d));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (passes & 2) {
    // Windowed: the grouped tile loop (which also serves ungrouped heads).
    auto kern = banded(p) ? (gproj ? bwd_col_wide_kernel<true, true, true> : bwd_col_wide_kernel<true, false, true>)
                : gproj ? (p.group > 1 ? bwd_col_wide_kernel<true, true> : bwd_col_wide_kernel<false, true>)
                        : (p.group > 1 ? bwd_col_wide_kernel<true, false> : bwd_col_wide_kernel<false, false>);
    const int bytes = gproj ? ColLayT<true>::bytes : ColLayT<false>::bytes;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(nb * p.BHkv), kThreads, bytes, st>>>(
        k, v, q, g, s, static_cast<__nv_bfloat16*>(dK), static_cast<__nv_bfloat16*>(dV), static_cast<int>(N), nb,
        static_cast<int>(p.BHkv), p.scale, c, p.causal, make_band(p, eff_window_tc(p), true), p.group, static_cast<int>(d));
    e = cudaGetLastError();
  }
  return e;
}

uint32_t tc_bwd_wide_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
