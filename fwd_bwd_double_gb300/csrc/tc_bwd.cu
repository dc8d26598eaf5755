// bf16 causal attention backward on sm_103a (tcgen05 + TMA), written once per
// output block: a row pass for dQ and a column pass for dK, dV.
//
// "Flash attention for trading models", "Backward pass: recompute instead of
// store": P is rebuilt from Q, K and the stored log-sum-exp; nothing N x N is
// stored.  With dP = dO V^T, D_i = dO_i . O_i and dS = P * (dP - D):
//   row pass    (CTA holds 128 query rows, streams 64-key blocks j <= i)
//               S = Q K_j^T, dP = dO V_j^T           (A, B from shared memory)
//               dQ += dS K_j                          (A = dS from TMEM, B = K_j MN-major)
//               writes dQ = s dQ once and the row statistics (L log2 e, D, rho), stored
//               negated and interleaved by row pairs for the column pass
//   column pass (CTA holds 128 keys, streams 64-query blocks i >= j)
//               S^T = K Q_i^T, dP^T = V dO_i^T        (transposed tiles: lanes = keys)
//               dV += P^T dO_i, dK += dS^T Q_i        (A from TMEM, B MN-major)
//               writes dK = s dK, dV once.
// GProj ("FlashAttention bf16 gradient and GProj", "How the zero sum turns into a
// false gradient"): the products see dS^ = bf16(dS) whose rows no longer sum to
// zero.  The row pass accumulates r_i = sum_j dS^_ij and sum_j P^_ij of the bf16
// values it feeds to the products, plus PK_i = P^ K; it writes
//   dQ_i = s (dS^ K - rho_i PK_i),  rho_i = r_i / sum_j P^_ij,
// i.e. the products of the projected row dS^_ij - rho_i P^_ij, which sums to zero.
// The key correction needs rho_i of complete rows, hence the separate column pass:
// it adds (-rho_i P^_ji) as a third A operand to the dK product.
//
// Roles: warps 0-7 compute (warp w owns TMEM lanes 32(w%4).., i.e. 32 rows, and
// half of each tile's 64 columns); warp 8 issues TMA loads; warp 9 allocates TMEM
// and issues the MMAs.  Score tiles are NB-buffered in TMEM so the MMAs of tile
// t+1 run while the compute warps turn tile t into dS.
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fbd {
namespace {

__device__ unsigned int g_err = 0;

constexpr int BM = 128;        // rows held by a CTA (queries, or keys in the column pass)
constexpr int BN = 64;         // rows of a streamed block
// Shared-memory stages of streamed tiles: deep enough that a tile is requested
// several tile-times before its MMA needs it (L2/HBM latency under load).
// At d = 256 one stage is all that fits beside the held block (64 KB a tile); the MMA
// warp then finishes each block's products before the next block's tiles (see below),
// and the row pass keeps K and V in buffers reloaded on their own (RowLay::SPLIT).
template <int D>
constexpr int stages() { return D == 64 ? 6 : D == 256 ? 1 : 4; }
constexpr int kCompute = 256;  // 8 compute warps
constexpr int kThreads = kCompute + 64;
constexpr float kLog2e = 1.4426950408889634f;

using tc::bf16_hi;
using tc::bf16_lo;
using tc::f;

// ================================================================ row pass
// With GProj at d = 256 the accumulators dQ and P^ K of the whole head dim would take
// 512 TMEM columns beside the tiles: each row block then runs as two CTAs, CTA h
// accumulating and writing output columns [DO h, DO h + DO) (DO = 128); both compute the
// full score tiles and the coefficient rho.
template <int D, int NB, bool GP>
struct RowLay {
  static constexpr int DO = (GP && D == 256) ? 128 : D;  // output columns a CTA accumulates
  // TMEM columns used (see below); at most 256 lets two CTAs share an SM, in which
  // case the ring is shortened so that both fit in shared memory.
  static constexpr int kCols = 2 * NB * BN + NB * BN / 2 + (GP ? NB * BN / 2 : 0) + DO + (GP ? DO : 0);
  static constexpr int kTmem = kCols <= 256 ? 256 : 512;
  static constexpr int kMinBlocks = kTmem == 256 ? 2 : 1;
  static constexpr int NS = kTmem == 256 ? 4 : stages<D>();
  // One stage (d = 256): K and V in buffers of their own, each reloaded as soon as the
  // products reading it are done (V after dP_j, K after S_j and the dQ product), V by a
  // second TMA warp, so that dP_{j+1} runs while K_{j+1} loads.
  static constexpr bool SPLIT = NS == 1;
  static constexpr int kThreadsRow = kThreads + (SPLIT ? 32 : 0);
  static constexpr int kHeld = BM * D * 2;
  static constexpr int kStream = BN * D * 2;
  static constexpr int oQ = 0, odO = kHeld, oK = 2 * kHeld, oV = oK + NS * kStream;
  static constexpr int oRed = oV + NS * kStream;  // float [6][BM]
  static constexpr int oBar = oRed + 6 * BM * 4;
  static constexpr int bytes = oBar + 256;
  static constexpr int cS = 0, cdP = NB * BN, cdS = 2 * NB * BN, cP = cdS + NB * BN / 2;
  static constexpr int cdQ = cP + (GP ? NB * BN / 2 : 0), cPK = cdQ + DO;
  static constexpr int cols = cPK + (GP ? DO : 0);
  static_assert(cols == kCols && cols <= 512, "TMEM budget");
};

// WIN: a banded causal mask is in force (bd: the sliding window and/or the document
// bounds); the other instances carry none of it.
template <int D, int NB, bool GP, bool WIN = false>
__global__ void __launch_bounds__(RowLay<D, NB, GP>::kThreadsRow, RowLay<D, NB, GP>::kMinBlocks)
    bwd_row_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
                   const float* __restrict__ lse, __nv_bfloat16* __restrict__ dQ, float4* __restrict__ ws, int N,
                   int Np, int nrb, int BH, float scale, float c, int causal, Band bd, int G, int dv) {
  using Lay = RowLay<D, NB, GP>;
  static_assert(NB == 1, "one score-tile buffer, released early");
  constexpr int NS = Lay::NS, DO = Lay::DO, HV = D / DO;  // HV CTAs per row block, one per output part
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* q_full = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
  uint64_t* full = q_full + 1;
  uint64_t* empty = full + NS;
  uint64_t* s_full = empty + NS;
  uint64_t* ds_ready = s_full + NB;     // dS (and P^) of the block in TMEM
  uint64_t* consumed = ds_ready + NB;   // the block's S, dP copied out: the tile columns are free
  uint64_t* out_done = consumed + 1;    // the block's dQ (and P^ K) products have read the operands
  uint64_t* acc_full = out_done + 1;
  // SPLIT: full[0] / empty[0] are K's (loaded / read by S_j and the dQ product), and
  uint64_t* v_full = acc_full + 1;   // V_j loaded
  uint64_t* v_empty = acc_full + 2;  // dP_j done: the V buffer free
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + (Lay::SPLIT ? 3 : 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(sm + Lay::oRed);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int opart = HV > 1 ? static_cast<int>(blockIdx.x) % HV : 0;  // output columns [DO opart, DO opart + DO)
  const tc::Order ord = tc::grid_order_at(static_cast<int>(blockIdx.x) / HV, BH, nrb);
  const int bh = ord.bh;
  const int rb = nrb - 1 - ord.k;  // heaviest row blocks first (within a group of slices)
  // key blocks j0 + j, j < nkv: those touching rows <= the last row (all key blocks when
  // not causal), from the first one a row sees under the banded mask bd
  const int j0 = (WIN && causal) ? bd.row_lo(bh, rb * BM) / BN : 0;
  const int lo_last = (WIN && causal) ? bd.row_lo(bh, min(rb * BM + BM - 1, N - 1)) : 0;
  const int nkv = (causal ? ((rb + 1) * BM + BN - 1) / BN : (N + BN - 1) / BN) - j0;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      ptx::mbar_init(&s_full[b], 1);
      ptx::mbar_init(&ds_ready[b], kCompute);
    }
    ptx::mbar_init(consumed, kCompute);
    ptx::mbar_init(out_done, 1);
    ptx::mbar_init(acc_full, 1);
    if constexpr (Lay::SPLIT) {
      ptx::mbar_init(v_full, 1);
      ptx::mbar_init(v_empty, 1);
    }
    *abort_flag = (ptx::smem_u32(sm) & 1023u) ? 1 : 0;
    if (*abort_flag) atomicOr(&g_err, FBD_ERR_TIMEOUT);
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(tmem_slot, Lay::kTmem);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::BoundedWait wait{abort_flag, &g_err};
  const bool ok = *abort_flag == 0;

  if (warp == 8) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0 && ok) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::mbar_expect_tx(q_full, 2 * Lay::kHeld);
      for (int cc = 0; cc < D / 64; ++cc) {
        ptx::tma_load_3d(sm + Lay::oQ + cc * BM * 128, &tmQ, q_full, cc * 64, rb * BM, bh);
        ptx::tma_load_3d(sm + Lay::odO + cc * BM * 128, &tmdO, q_full, cc * 64, rb * BM, bh);
      }
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS;
        if (j >= NS) wait(&empty[s], ((j / NS) - 1) & 1);
        ptx::mbar_expect_tx(&full[s], (Lay::SPLIT ? 1 : 2) * Lay::kStream);
        for (int cc = 0; cc < D / 64; ++cc) {
          ptx::tma_load_3d(sm + Lay::oK + s * Lay::kStream + cc * BN * 128, &tmK, &full[s], cc * 64, (j0 + j) * BN,
                           bh / G);
          if constexpr (!Lay::SPLIT)
            ptx::tma_load_3d(sm + Lay::oV + s * Lay::kStream + cc * BN * 128, &tmV, &full[s], cc * 64,
                             (j0 + j) * BN, bh / G);
        }
      }
      for (int j = (nkv > NS ? nkv - NS : 0); j < nkv; ++j) wait(&empty[j % NS], (j / NS) & 1);
    }
  } else if (Lay::SPLIT && warp == kThreads / 32) {
    // ------------------------------------------------- V loader (one stage)
    if (lane == 0 && ok) {
      for (int j = 0; j < nkv; ++j) {
        if (j >= 1) wait(v_empty, (j - 1) & 1);  // dP_{j-1} has read the V buffer
        ptx::mbar_expect_tx(v_full, Lay::kStream);
        for (int cc = 0; cc < D / 64; ++cc)
          ptx::tma_load_3d(sm + Lay::oV + cc * BN * 128, &tmV, v_full, cc * 64, (j0 + j) * BN, bh / G);
      }
      if (nkv > 0) wait(v_empty, (nkv - 1) & 1);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idS = ptx::idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idQ = ptx::idesc_bf16(BM, DO, 0, 1);
      const uint32_t sQ = ptx::smem_u32(sm + Lay::oQ), sdO = ptx::smem_u32(sm + Lay::odO);
      const uint32_t sK = ptx::smem_u32(sm + Lay::oK), sV = ptx::smem_u32(sm + Lay::oV);
      const uint32_t po = static_cast<uint32_t>(opart * (DO / 64) * BN * 128);  // this CTA's column slabs
      auto products = [&](int t) {  // dQ (+ P^ K) of tile t, then release its stage
        const int b = t % NB, s = t % NS;
        wait(&ds_ready[b], (t / NB) & 1);
        ptx::tc_fence_after();
        const uint32_t kt = sK + s * Lay::kStream + po;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t bd = tc::mnmajor_desc(kt, BN, k);
          ptx::mma_ts_e(tmem + Lay::cdQ, tmem + Lay::cdS + b * (BN / 2) + k * 8, bd, idQ, (t > 0 || k > 0));
          if constexpr (GP)
            ptx::mma_ts_e(tmem + Lay::cPK, tmem + Lay::cP + b * (BN / 2) + k * 8, bd, idQ, (t > 0 || k > 0));
        }
        ptx::mma_commit_e(&empty[s]);
        ptx::mma_commit_e(out_done);
      };
      // Block j's tiles go into the columns block j-1's tiles left as soon as the
      // compute warps have copied those out (`consumed`), ahead of block j-1's products.
      // With a single stage the block's own products come first (they read K_j, which
      // the next block's load replaces); V_{j+1} is loaded as soon as dP_j is done, so
      // dP_{j+1} runs on the pipe while K_{j+1} comes in.
      wait(q_full, 0);
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS, b = j % NB;
        const uint32_t kt = sK + s * Lay::kStream, vt = sV + s * Lay::kStream;
        if constexpr (Lay::SPLIT) {
          // dP_j first (V_j came in while the previous block's products ran), then S_j once
          // K_j has replaced K_{j-1}.
          if (j > 0) wait(consumed, (j - 1) & 1);
          wait(v_full, j & 1);
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss_e(tmem + Lay::cdP + b * BN, tc::kmajor_desc(sdO, BM, kk), tc::kmajor_desc(vt, BN, kk), idS,
                          kk > 0);
          ptx::mma_commit_e(v_empty);
          wait(&full[s], (j / NS) & 1);
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss_e(tmem + Lay::cS + b * BN, tc::kmajor_desc(sQ, BM, kk), tc::kmajor_desc(kt, BN, kk), idS,
                          kk > 0);
        } else {
          wait(&full[s], (j / NS) & 1);
          if (j > 0) wait(consumed, (j - 1) & 1);
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss_e(tmem + Lay::cS + b * BN, tc::kmajor_desc(sQ, BM, kk), tc::kmajor_desc(kt, BN, kk), idS,
                          kk > 0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss_e(tmem + Lay::cdP + b * BN, tc::kmajor_desc(sdO, BM, kk), tc::kmajor_desc(vt, BN, kk), idS,
                          kk > 0);
        }
        ptx::mma_commit_e(&s_full[b]);
        if constexpr (NS == 1) {
          products(j);
        } else if (j > 0) {
          products(j - 1);
        }
      }
      if (NS > 1 && nkv > 0) products(nkv - 1);
      ptx::mma_commit_e(acc_full);
    }
  } else {
    // ------------------------------------------------------------- compute
    const int qd = warp & 3, hf = warp >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>(qd * 32) << 16;
    const int64_t row = static_cast<int64_t>(rb) * BM + r;
    const bool live = row < N;
    const size_t rowoff = (static_cast<size_t>(bh) * N + row) * dv;  // rows of dv <= D columns
    float part = 0.f;
    if (live) {  // this thread's half of D_r = dO_r . O_r
      const uint4* po = reinterpret_cast<const uint4*>(O + rowoff + hf * (D / 2));
      const uint4* pg = reinterpret_cast<const uint4*>(dO + rowoff + hf * (D / 2));
#pragma unroll
      for (int u = 0; u < D / 16; ++u) {
        if (hf * (D / 2) + 8 * u >= dv) break;  // padding columns
        const uint4 a = po[u], g = pg[u];
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) part += bf16_lo(aw[e]) * bf16_lo(gw[e]) + bf16_hi(aw[e]) * bf16_hi(gw[e]);
      }
    }
    red[hf * BM + r] = part;
    tc::named_sync(1, kCompute);
    const float Dr = red[r] + red[BM + r];
    const float L2 = live ? lse[static_cast<size_t>(bh) * N + row] * kLog2e : 0.f;
    uint64_t accR = 0, accP = 0;  // GProj: sums of the bf16 dS and P fed to the products
    const uint64_t c2 = tc::pk2f(c, c), nL2 = tc::pk2f(-L2, -L2), nD2 = tc::pk2f(-Dr, -Dr);
    const int c0 = hf * (BN / 2);
    const int lo_row = (WIN && causal) ? bd.row_lo(bh, row) : 0;
    for (int j = 0; j < nkv; ++j) {
      const int b = j % NB;
      wait(&s_full[b], (j / NB) & 1);
      ptx::tc_fence_after();
      uint32_t sv[32], pv[32];
      ptx::tmem_ld32(tmem + Lay::cS + b * BN + c0 + lo, sv);
      ptx::tmem_ld32(tmem + Lay::cdP + b * BN + c0 + lo, pv);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(consumed);  // the MMA warp may now compute the next block's tiles here
      const int kb = j0 + j;
      const int krel = kb * BN + c0 - rb * BM;  // key of my column 0 minus the block's first row
      // last and first visible key of this row, relative to my column 0
      const int klim = causal ? r - krel : N - 1 - (kb * BN + c0);
      const int klo = (WIN && causal) ? lo_row - (kb * BN + c0) : 0;
      uint32_t dsk[16], pk[16];
      auto block = [&](auto masked) {
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const float2 arg = tc::unpk2(tc::fma2(tc::pk2(sv[t], sv[t + 1]), c2, nL2));
          float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
          if constexpr (decltype(masked)::value) {
            if (t > klim || t < klo) p0 = 0.f;
            if (t + 1 > klim || t + 1 < klo) p1 = 0.f;
          }
          const float2 ds = tc::unpk2(tc::mul2(tc::pk2f(p0, p1), tc::add2(tc::pk2(pv[t], pv[t + 1]), nD2)));
          dsk[t >> 1] = ptx::pack_bf16(ds.x, ds.y);
          if constexpr (GP) {
            pk[t >> 1] = ptx::pack_bf16(p0, p1);
            accR = tc::add2(accR, tc::bf2_to_f2(dsk[t >> 1]));
            accP = tc::add2(accP, tc::bf2_to_f2(pk[t >> 1]));
          }
        }
      };
      // the mask reaches into this thread's columns: past the row (causal), below the
      // window of the block's last row, or past N
      if (causal ? (krel + 31 > 0 || (WIN && kb * BN + c0 < lo_last)) : kb * BN + c0 + 32 > N)
        block(std::true_type{});
      else
        block(std::false_type{});
      if (j > 0) wait(out_done, (j - 1) & 1);  // block j-1's products have read dS (and P^)
      ptx::tmem_st16(tmem + Lay::cdS + b * (BN / 2) + c0 / 2 + lo, dsk);
      if constexpr (GP) ptx::tmem_st16(tmem + Lay::cP + b * (BN / 2) + c0 / 2 + lo, pk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ds_ready[b]);
    }
    float rho = 0.f;
    if constexpr (GP) {
      const float2 vr = tc::unpk2(accR), vp = tc::unpk2(accP);
      red[2 * BM + hf * BM + r] = vr.x + vr.y;
      red[4 * BM + hf * BM + r] = vp.x + vp.y;
      tc::named_sync(1, kCompute);
      rho = (red[2 * BM + r] + red[3 * BM + r]) / (red[4 * BM + r] + red[5 * BM + r]);
    }
    wait(acc_full, 0);
    ptx::tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < DO / 2; cc += 32) {
      uint32_t a[32], pkv[32];
      ptx::tmem_ld32(tmem + Lay::cdQ + hf * (DO / 2) + cc + lo, a);
      if constexpr (GP) ptx::tmem_ld32(tmem + Lay::cPK + hf * (DO / 2) + cc + lo, pkv);
      ptx::tmem_wait_ld();
      const int col = opart * DO + hf * (DO / 2) + cc;  // first of the 32 output columns
      if (live && col < dv) {
        uint32_t o[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          float v0 = f(a[t]), v1 = f(a[t + 1]);
          if constexpr (GP) {
            v0 -= rho * f(pkv[t]);
            v1 -= rho * f(pkv[t + 1]);
          }
          o[t >> 1] = ptx::pack_bf16(scale * v0, scale * v1);
        }
        uint4* dst = reinterpret_cast<uint4*>(dQ + rowoff + col);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
      }
    }
    if (hf == 0 && opart == 0 && row < Np) {  // row statistics, negated, pair-interleaved (see the column pass)
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
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Lay::kTmem);
  }
}

// ============================================================= column pass
// At d = 256 the accumulators dV, dK of the whole head dim would take 512 TMEM columns
// beside the tiles: each key block runs as two CTAs, CTA h accumulating and writing output
// columns [DO h, DO h + DO) (DO = 128); both compute the full score tiles.
template <int D, int NB, bool GP>
struct ColLay {
  static constexpr int DO = D == 256 ? 128 : D;  // output columns a CTA accumulates
  static constexpr int NS = stages<D>();
  static constexpr int kHeld = BM * D * 2;
  static constexpr int kStream = BN * D * 2;
  static constexpr int kStat = BN * 16;
  static constexpr int oK = 0, oV = kHeld, oQ = 2 * kHeld, odO = oQ + NS * kStream, oSt = odO + NS * kStream;
  static constexpr int oBar = oSt + NS * kStat;
  static constexpr int bytes = oBar + 256;
  static constexpr int cS = 0, cdP = NB * BN, cP = 2 * NB * BN, cdS = cP + NB * BN / 2, cG = cdS + NB * BN / 2;
  static constexpr int cdV = cG + (GP ? NB * BN / 2 : 0), cdK = cdV + DO;
  static constexpr int cols = cdK + DO;
  static_assert(cols <= 512, "TMEM budget");
};

// GR: grouped key/value heads (G > 1).  The G == 1 instance keeps the plain tile loop.
template <int D, int NB, bool GP, bool GR, bool WIN = false>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_col_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmSt, __nv_bfloat16* __restrict__ dK,
                   __nv_bfloat16* __restrict__ dV, int N, int BHkv, float scale, float c, int causal, Band bd, int G,
                   int dv) {
  using Lay = ColLay<D, NB, GP>;
  static_assert(NB == 1, "one score-tile buffer, released early");
  constexpr int NS = Lay::NS, DO = Lay::DO, HV = D / DO;  // HV CTAs per key block, one per output part
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* k_full = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
  uint64_t* full = k_full + 1;
  uint64_t* empty = full + NS;
  uint64_t* s_full = empty + NS;
  uint64_t* ds_ready = s_full + NB;     // P, dS (and the GProj operand) of the block in TMEM
  uint64_t* consumed = ds_ready + NB;   // the block's S^T, dP^T copied out: the tile columns are free
  uint64_t* out_done = consumed + 1;    // the block's dV, dK products have read the operand columns
  uint64_t* acc_full = out_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + BM - 1) / BM;
  const int part = HV > 1 ? static_cast<int>(blockIdx.x) % HV : 0;  // output columns [DO part, DO part + DO)
  const tc::Order ord = tc::grid_order_at(static_cast<int>(blockIdx.x) / HV, BHkv, nkb);
  const int kvh = ord.bh;  // key/value slice; its G query slices are kvh * G + h, h < G
  const int kb = ord.k;  // first key blocks have the most rows: first
  const int nq = (N + BN - 1) / BN;
  const int i0 = causal ? (kb * BM) / BN : 0;         // first query block with a query >= first key
  // query blocks per query slice: up to the last query any key of the block sees (bd.key_hi)
  const int ntile = ((WIN && causal) ? bd.key_hi(kvh, min(kb * BM + BM - 1, N - 1)) / BN + 1 : nq) - i0;
  const int hi_first = (WIN && causal) ? bd.key_hi(kvh, kb * BM) : 0;  // the block's first key's last query
  const int nt = GR ? G * ntile : ntile;              // tiles t = h * ntile + (i - i0), one dK, dV

  if (threadIdx.x == 0) {
    ptx::mbar_init(k_full, 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      ptx::mbar_init(&s_full[b], 1);
      ptx::mbar_init(&ds_ready[b], kCompute);
    }
    ptx::mbar_init(consumed, kCompute);
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
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmdO);
      ptx::prefetch_tmap(&tmSt);
      ptx::mbar_expect_tx(k_full, 2 * Lay::kHeld);
      for (int cc = 0; cc < D / 64; ++cc) {
        ptx::tma_load_3d(sm + Lay::oK + cc * BM * 128, &tmK, k_full, cc * 64, kb * BM, kvh);
        ptx::tma_load_3d(sm + Lay::oV + cc * BM * 128, &tmV, k_full, cc * 64, kb * BM, kvh);
      }
      for (int t = 0; t < nt; ++t) {
        const int h = GR ? t / ntile : 0, s = t % NS, i = i0 + t - h * ntile, bh = GR ? kvh * G + h : kvh;
        if (t >= NS) wait(&empty[s], ((t / NS) - 1) & 1);
        ptx::mbar_expect_tx(&full[s], 2 * Lay::kStream + Lay::kStat);
        for (int cc = 0; cc < D / 64; ++cc) {
          ptx::tma_load_3d(sm + Lay::oQ + s * Lay::kStream + cc * BN * 128, &tmQ, &full[s], cc * 64, i * BN, bh);
          ptx::tma_load_3d(sm + Lay::odO + s * Lay::kStream + cc * BN * 128, &tmdO, &full[s], cc * 64, i * BN, bh);
        }
        ptx::tma_load_3d(sm + Lay::oSt + s * Lay::kStat, &tmSt, &full[s], 0, i * BN, bh);
      }
      for (int t = (nt > NS ? nt - NS : 0); t < nt; ++t) wait(&empty[t % NS], (t / NS) & 1);
    }
  } else if (warp == 9) {
    if (ok) {  // all 32 lanes; one elected lane issues each MMA and commit
      constexpr uint32_t idS = ptx::idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idKV = ptx::idesc_bf16(BM, DO, 0, 1);
      const uint32_t sK = ptx::smem_u32(sm + Lay::oK), sV = ptx::smem_u32(sm + Lay::oV);
      const uint32_t sQ = ptx::smem_u32(sm + Lay::oQ), sdO = ptx::smem_u32(sm + Lay::odO);
      const uint32_t po = static_cast<uint32_t>(part * (DO / 64) * BN * 128);  // this CTA's column slabs
      auto products = [&](int t) {
        const int b = t % NB, s = t % NS;
        wait(&ds_ready[b], (t / NB) & 1);
        ptx::tc_fence_after();
        const uint32_t qt = sQ + s * Lay::kStream + po, gt = sdO + s * Lay::kStream + po;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          ptx::mma_ts_e(tmem + Lay::cdV, tmem + Lay::cP + b * (BN / 2) + k * 8, tc::mnmajor_desc(gt, BN, k), idKV,
                      (t > 0 || k > 0));
          const uint64_t bq = tc::mnmajor_desc(qt, BN, k);
          ptx::mma_ts_e(tmem + Lay::cdK, tmem + Lay::cdS + b * (BN / 2) + k * 8, bq, idKV, (t > 0 || k > 0));
          if constexpr (GP) ptx::mma_ts_e(tmem + Lay::cdK, tmem + Lay::cG + b * (BN / 2) + k * 8, bq, idKV, 1u);
        }
        ptx::mma_commit_e(&empty[s]);
        ptx::mma_commit_e(out_done);
      };
      // Block t's tiles go into the columns block t-1's tiles left as soon as the
      // compute warps have copied those out (`consumed`), ahead of block t-1's products.
      wait(k_full, 0);
      for (int t = 0; t < nt; ++t) {
        const int s = t % NS, b = t % NB;
        wait(&full[s], (t / NS) & 1);
        if (t > 0) wait(consumed, (t - 1) & 1);
        ptx::tc_fence_after();
        const uint32_t qt = sQ + s * Lay::kStream, gt = sdO + s * Lay::kStream;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tmem + Lay::cS + b * BN, tc::kmajor_desc(sK, BM, kk), tc::kmajor_desc(qt, BN, kk), idS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tmem + Lay::cdP + b * BN, tc::kmajor_desc(sV, BM, kk), tc::kmajor_desc(gt, BN, kk), idS,
                      kk > 0);
        ptx::mma_commit_e(&s_full[b]);
        if constexpr (NS == 1) {  // one stage: the block's products before the next block's load
          products(t);
        } else if (t > 0) {
          products(t - 1);
        }
      }
      if (NS > 1 && nt > 0) products(nt - 1);
      ptx::mma_commit_e(acc_full);
    }
  } else {
    const int qd = warp & 3, hf = warp >> 2;
    const int r = qd * 32 + lane;  // key row within the block (TMEM lane)
    const uint32_t lo = static_cast<uint32_t>(qd * 32) << 16;
    const int key = kb * BM + r;
    const int c0 = hf * (BN / 2);
    const uint64_t c2 = tc::pk2f(c, c);
    const int khi = (WIN && causal) ? bd.key_hi(kvh, key) : 0;  // the last query this key is seen by
    for (int t = 0; t < nt; ++t) {
      const int s = t % NS, b = t % NB, i = GR ? i0 + t % ntile : i0 + t;
      wait(&s_full[b], (t / NB) & 1);
      ptx::tc_fence_after();
      uint32_t sv[32], pv[32];
      ptx::tmem_ld32(tmem + Lay::cS + b * BN + c0 + lo, sv);
      ptx::tmem_ld32(tmem + Lay::cdP + b * BN + c0 + lo, pv);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(consumed);  // the MMA warp may now compute the next block's tiles here
      // Row statistics of the 64 queries, pair-interleaved: float4 2m = (-L2, -L2', -D, -D'),
      // float4 2m+1 = (-rho, -rho', 0, 0) of queries 2m, 2m+1 of the block.
      const float4* st = reinterpret_cast<const float4*>(sm + Lay::oSt + s * Lay::kStat) + c0;
      const int qbase = i * BN + c0;
      uint32_t pk[16], dk[16], gk[16];
      auto block = [&](auto masked) {
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          const float4 A = st[u];
          const float2 arg = tc::unpk2(tc::fma2(tc::pk2(sv[u], sv[u + 1]), c2, tc::pk2f(A.x, A.y)));
          float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
          if constexpr (decltype(masked)::value) {
            const int q0 = qbase + u;
            if ((causal && (q0 < key || (WIN && q0 > khi))) || q0 >= N) p0 = 0.f;
            if ((causal && (q0 + 1 < key || (WIN && q0 + 1 > khi))) || q0 + 1 >= N) p1 = 0.f;
          }
          const float2 ds =
              tc::unpk2(tc::mul2(tc::pk2f(p0, p1), tc::add2(tc::pk2(pv[u], pv[u + 1]), tc::pk2f(A.z, A.w))));
          pk[u >> 1] = ptx::pack_bf16(p0, p1);
          dk[u >> 1] = ptx::pack_bf16(ds.x, ds.y);
          if constexpr (GP) {
            const float4 Bs = st[u + 1];
            const float2 g = tc::unpk2(tc::mul2(tc::pk2f(Bs.x, Bs.y), tc::bf2_to_f2(pk[u >> 1])));
            gk[u >> 1] = ptx::pack_bf16(g.x, g.y);
          }
        }
      };
      // causal mask (first blocks), past the window of the block's first key, or past N (last block)
      if ((causal && (qbase < kb * BM + BM || (WIN && qbase + 31 > hi_first))) || qbase + 32 > N)
        block(std::true_type{});
      else
        block(std::false_type{});
      if (t > 0) wait(out_done, (t - 1) & 1);  // block t-1's products have read P, dS
      ptx::tmem_st16(tmem + Lay::cP + b * (BN / 2) + c0 / 2 + lo, pk);
      ptx::tmem_st16(tmem + Lay::cdS + b * (BN / 2) + c0 / 2 + lo, dk);
      if constexpr (GP) ptx::tmem_st16(tmem + Lay::cG + b * (BN / 2) + c0 / 2 + lo, gk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ds_ready[b]);
    }
    wait(acc_full, 0);
    ptx::tc_fence_after();
    const bool live = key < N;
    const size_t rowoff = (static_cast<size_t>(kvh) * N + key) * dv;
#pragma unroll
    for (int cc = 0; cc < DO / 2; cc += 32) {
      uint32_t a[32], g[32];
      ptx::tmem_ld32(tmem + Lay::cdV + hf * (DO / 2) + cc + lo, a);
      ptx::tmem_ld32(tmem + Lay::cdK + hf * (DO / 2) + cc + lo, g);
      ptx::tmem_wait_ld();
      const int col = part * DO + hf * (DO / 2) + cc;  // first of the 32 output columns
      if (live && col < dv) {
        uint32_t ov[16], ok2[16];
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          ov[u >> 1] = ptx::pack_bf16(f(a[u]), f(a[u + 1]));
          ok2[u >> 1] = ptx::pack_bf16(scale * f(g[u]), scale * f(g[u + 1]));
        }
        uint4* dvp = reinterpret_cast<uint4*>(dV + rowoff + col);
        uint4* dk2 = reinterpret_cast<uint4*>(dK + rowoff + col);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          dvp[u] = make_uint4(ov[4 * u], ov[4 * u + 1], ov[4 * u + 2], ov[4 * u + 3]);
          dk2[u] = make_uint4(ok2[4 * u], ok2[4 * u + 1], ok2[4 * u + 2], ok2[4 * u + 3]);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, int NBR, int NBC, bool GP>
cudaError_t launch(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes, cudaStream_t st) {
  alignas(64) CUtensorMap q128, do128, k64, v64, k128, v128, q64, do64, s64;
  const int64_t N = p.N, BH = p.BH, Np = (p.N + 1) & ~static_cast<int64_t>(1);
  const int64_t d = p.d;  // <= D; TMA zero-fills the padding columns d .. D-1
  if (!make_tmap_bf16(&q128, Q, N, d, BH, BM) || !make_tmap_bf16(&do128, dO, N, d, BH, BM) ||
      !make_tmap_bf16(&k64, K, N, d, p.BHkv, BN) || !make_tmap_bf16(&v64, V, N, d, p.BHkv, BN) ||
      !make_tmap_bf16(&k128, K, N, d, p.BHkv, BM) || !make_tmap_bf16(&v128, V, N, d, p.BHkv, BM) ||
      !make_tmap_bf16(&q64, Q, N, d, BH, BN) || !make_tmap_bf16(&do64, dO, N, d, BH, BN) ||
      !make_tmap_stats(&s64, ws, Np, BH, BN))
    return cudaErrorInvalidValue;
  const float c = p.scale * kLog2e;
  const int nrb = static_cast<int>((N + BM - 1) / BM);
  if (passes & 1) {
    using Lay = RowLay<D, NBR, GP>;
    auto kern = banded(p) ? bwd_row_kernel<D, NBR, GP, true> : bwd_row_kernel<D, NBR, GP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::bytes);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(nrb * BH * (D / Lay::DO)), Lay::kThreadsRow, Lay::bytes, st>>>(
        q128, do128, k64, v64, static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), lse,
        static_cast<__nv_bfloat16*>(dQ), ws, static_cast<int>(N), static_cast<int>(Np), nrb, static_cast<int>(BH),
        p.scale, c, p.causal, make_band(p, eff_window_tc(p), false), p.group, static_cast<int>(d));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (passes & 2) {
    using Lay = ColLay<D, NBC, GP>;
    // Windowed: the grouped tile loop (which also serves ungrouped heads).
    auto kern = banded(p) ? bwd_col_kernel<D, NBC, GP, true, true>
                : p.group > 1 ? bwd_col_kernel<D, NBC, GP, true> : bwd_col_kernel<D, NBC, GP, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::bytes);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(nrb * p.BHkv * (D / Lay::DO)), kThreads, Lay::bytes, st>>>(
        k128, v128, q64, do64, s64, static_cast<__nv_bfloat16*>(dK), static_cast<__nv_bfloat16*>(dV),
        static_cast<int>(N), static_cast<int>(p.BHkv), p.scale, c, p.causal, make_band(p, eff_window_tc(p), true),
        p.group, static_cast<int>(d));
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t tc_bwd(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* lse, void* dQ, void* dK, void* dV, int gproj, float4* ws, int passes,
                   cudaStream_t st) {
  // d = 32 runs the d = 64 kernels and d = 96 the d = 128 ones, zero-padded in shared memory.
  // d <= 64, with or without GProj: the 128-wide kernels.
  if (p.d <= 64) return tc_bwd_wide(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st, gproj != 0);
  // d = 256: both passes here (one stage; the column pass in two output halves, and with
  // GProj the row pass too).
  if (p.d > 128) {
    if (gproj) return launch<256, 1, 1, true>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st);
    return launch<256, 1, 1, false>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st);
  }
  if (gproj) return launch<128, 1, 1, true>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st);
  // d = 96, 128 without GProj: the 128-wide row pass, then this file's column pass
  // (both use the same pair-interleaved row statistics).
  if (passes & 1) {
    const cudaError_t e = tc_bwd_wide(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, 1, st);
    if (e != cudaSuccess) return e;
  }
  if (!(passes & 2)) return cudaSuccess;
  return launch<128, 1, 1, false>(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, 2, st);
}

uint32_t tc_bwd_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
