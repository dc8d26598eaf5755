// bf16 attention backward in one pass over key blocks (d <= 64, without GProj).
//
// "Flash attention for trading models", "Backward pass: recompute instead of store":
// P = 2^(S s log2 e - L log2 e), dP = dO V^T, D_i = sum_k dO_ik O_ik, dS = P (dP - D);
// dQ = s dS K, dK = s dS^T Q, dV = P^T dO.  One CTA holds a block of 128 keys and streams
// the blocks of 128 queries that see it (section "FA2: parallelism": the work is split
// over key blocks and the query gradient is summed across them).  Per query block the
// tensor cores run each of the five contractions of the definition once:
//   S^T = K Q^T,  dP^T = V dO^T       tile products (M = N = 128), K and V held in shared
//                                     memory, the tiles in TMEM, released early
//   dV += P^T dO                      A = P^T (bf16) in TMEM
//   dK += dS^T Q                      A = dS^T from a shared-memory tile ...
//   dQ_i = dS K                       ... the same tile read M-major as dS
// dK and dV accumulate in TMEM for the whole block and are written once.  The block's
// share of dQ_i (128 x 64 fp32) is copied from TMEM into the stage that held Q_i and
// dO_i (free once the products that read them are done), after the next block's
// operands are released, and reduce-added into an fp32 accumulator by a TMA tensor
// reduce; the TMA warp then refills the stage.  The accumulator receives its partial
// sums in the order the key blocks reach it, so dQ can differ between runs in its last
// bits; dK and dV are the same bits every run.
//
// Launches: bwd_prep_kernel (D_i, the pair-interleaved negated row statistics the
// column passes read, the zeroed accumulator), bwd_fused_kernel, bwd_dq_kernel
// (dQ = bf16(s acc), each element written once).
//
// Warps 0-15 compute (warp w: TMEM lanes 32(w%4).., tile columns 32(w/4)..), warp 16
// issues the TMA loads and the dQ reduces, warp 17 the tile MMAs, warp 18 the output
// MMAs (both issue through elect.sync from the whole warp).
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fbd {
namespace {

__device__ unsigned int g_err = 0;

constexpr int D = 64;
constexpr int BW = 128;        // held key block and streamed query block rows
constexpr int NS = 4;          // stages of streamed blocks
constexpr int kCW = 16;        // compute warps
constexpr int kCompute = kCW * 32;
constexpr int kThreads = kCompute + 96;  // + TMA/reduce warp, tile-MMA warp, output-MMA warp
constexpr int kC = 32;         // tile columns per compute thread
constexpr int DG = D / 4;      // output columns per compute thread
constexpr int kTile = BW * D * 2;  // 16 KB
constexpr float kLog2e = 1.4426950408889634f;

struct Lay {
  static constexpr int kStat = BW * 16;
  // Q_i, dO_i (after block i's products, its fp32 dQ share: two boxes of 32 columns,
  // until the reduce has read it), statistics
  static constexpr int kStage = 2 * kTile + kStat;
  static constexpr int oK = 0, oV = kTile;
  static constexpr int odS = 2 * kTile;  // dS: 2 slabs (queries 0-63, 64-127) of 128 key lines
  static constexpr int oStage = odS + 2 * kTile;
  static constexpr int oBar = oStage + NS * kStage;
  static constexpr int bytes = oBar + 256;
  // TMEM columns: S^T, dP^T (fp32 tiles), P^T (bf16 pairs), dQ_i, dV, dK (fp32).
  static constexpr int cS = 0, cdP = 128, cP = 256, cdQ = 320, cdV = 384, cdK = 448;
};
static_assert(Lay::bytes <= 232448 && Lay::oStage % 1024 == 0 && Lay::kStage % 1024 == 0, "fused layout");

struct Bars {
  uint64_t* held_full;
  uint64_t* full;      // [NS] stage loaded
  uint64_t* s_full;    // S^T, dP^T of the block in TMEM
  uint64_t* consumed;  // ... copied into the compute registers
  uint64_t* ready;     // P^T in TMEM and dS in shared memory
  uint64_t* dq_full;   // the block's three output products finished (dQ_i in TMEM, P^T, dS read)
  uint64_t* dq_empty;  // dQ_i copied out of TMEM (the next block's dQ product may start)
  uint64_t* stg_full;  // [NS] dQ_i staged in its stage (one barrier per stage: the compute
                       // warps cannot run a full ring ahead of the reduces, so no phase of
                       // it completes twice before its wait)
  uint64_t* acc_full;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  __device__ explicit Bars(uint8_t* b) {
    held_full = reinterpret_cast<uint64_t*>(b);
    full = held_full + 1;
    s_full = full + NS;
    consumed = s_full + 1;
    ready = consumed + 1;
    dq_full = ready + 1;
    dq_empty = dq_full + 1;
    stg_full = dq_empty + 1;
    acc_full = stg_full + NS;
    tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  }
};

// Byte offset of (row, 16-byte chunk) in a 128-byte-swizzled tile of 128-byte lines
// (the layout a TMA box with 128-byte swizzle reads and writes; tile 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// GR: grouped key/value heads (G > 1); WIN: a banded causal mask is in force (bd: the
// sliding window and/or the document bounds).
template <bool GR, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_fused_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmSt, const __grid_constant__ CUtensorMap tmAcc,
                     __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, int N, int nb, int BHkv,
                     float scale, float c, int causal, Band bd, int G, int dv) {
  extern __shared__ __align__(1024) uint8_t sm[];
  Bars br(sm + Lay::oBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Order ord = tc::grid_order(BHkv, nb);
  const int kvh = ord.bh;          // key/value slice; its G query slices are kvh * G + h, h < G
  const int kb = ord.k;            // first key blocks have the most query blocks: first
  const int i0 = causal ? kb : 0;  // first query block that sees this key block
  // query blocks per query slice: up to the last query any key of the block sees (the
  // banded mask bd: queries i <= bd.key_hi(key))
  const int ntile = ((WIN && causal) ? bd.key_hi(kvh, min(kb * BW + BW - 1, N - 1)) / BW + 1 : nb) - i0;
  const int hi_first = (WIN && causal) ? bd.key_hi(kvh, kb * BW) : 0;  // the block's first key's last query
  const int nt = GR ? G * ntile : ntile;  // tiles t = h * ntile + (i - i0)

  if (threadIdx.x == 0) {
    ptx::mbar_init(br.held_full, 1);
    for (int s = 0; s < NS; ++s) ptx::mbar_init(&br.full[s], 1);
    ptx::mbar_init(br.s_full, 1);
    ptx::mbar_init(br.consumed, kCompute);
    ptx::mbar_init(br.ready, kCompute);
    ptx::mbar_init(br.dq_full, 1);
    ptx::mbar_init(br.dq_empty, kCompute);
    for (int s = 0; s < NS; ++s) ptx::mbar_init(&br.stg_full[s], kCompute);
    ptx::mbar_init(br.acc_full, 1);
    *br.abort_flag = (ptx::smem_u32(sm) & 1023u) ? 1 : 0;
    if (*br.abort_flag) atomicOr(&g_err, FBD_ERR_TIMEOUT);
    ptx::fence_mbar_init();
  }
  if (warp == kCW + 1) {
    ptx::tmem_alloc(br.tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *br.tmem_slot;
  const ptx::BoundedWait wait{br.abort_flag, &g_err};
  const bool ok = *br.abort_flag == 0;
  auto tile_at = [&](int t, int& bh, int& i) {
    const int h = GR ? t / ntile : 0;
    bh = GR ? kvh * G + h : kvh;
    i = i0 + t - h * ntile;
  };

  if (warp == kCW) {
    // ------------------------------------------------ TMA loads and dQ reduces
    if (lane == 0 && ok) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmdO);
      ptx::prefetch_tmap(&tmSt);
      ptx::prefetch_tmap(&tmAcc);
      ptx::mbar_expect_tx(br.held_full, 2 * kTile);
      ptx::tma_load_3d(sm + Lay::oK, &tmK, br.held_full, 0, kb * BW, kvh);
      ptx::tma_load_3d(sm + Lay::oV, &tmV, br.held_full, 0, kb * BW, kvh);
      auto load = [&](int t) {
        int bh, i;
        tile_at(t, bh, i);
        const int s = t % NS;
        uint8_t* st = sm + Lay::oStage + s * Lay::kStage;
        ptx::mbar_expect_tx(&br.full[s], 2 * kTile + Lay::kStat);
        ptx::tma_load_3d(st, &tmQ, &br.full[s], 0, i * BW, bh);
        ptx::tma_load_3d(st + kTile, &tmdO, &br.full[s], 0, i * BW, bh);
        ptx::tma_load_3d(st + 2 * kTile, &tmSt, &br.full[s], 0, i * BW, bh);
      };
      for (int t = 0; t < nt && t < NS; ++t) load(t);
      for (int t = 0; t < nt; ++t) {
        // dQ_t staged in its stage: reduce-add the two 32-column boxes, then refill the stage.
        if (!wait(&br.stg_full[t % NS], (t / NS) & 1)) break;
        int bh, i;
        tile_at(t, bh, i);
        const uint8_t* st = sm + Lay::oStage + (t % NS) * Lay::kStage;
        ptx::tma_reduce_add_3d(&tmAcc, st, 0, i * BW, bh);
        ptx::tma_reduce_add_3d(&tmAcc, st + kTile, 32, i * BW, bh);
        ptx::bulk_commit_group();
        ptx::bulk_wait_group_read0();  // the stage's bytes have been read
        if (t + NS < nt) load(t + NS);
      }
      ptx::bulk_wait_group0();  // every reduce performed before the CTA ends
    }
  } else if (warp == kCW + 1) {
    // ---------------------------------------------------------- tile MMAs
    if (ok) {
      constexpr uint32_t idS = ptx::idesc_bf16(BW, BW, 0, 0);
      const uint64_t dKk = tc::kmajor_desc(ptx::smem_u32(sm + Lay::oK), BW, 0);
      const uint64_t dVk = tc::kmajor_desc(ptx::smem_u32(sm + Lay::oV), BW, 0);
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage);
      const uint64_t dQk = tc::kmajor_desc(sSt, BW, 0), ddOk = tc::kmajor_desc(sSt + kTile, BW, 0);
      const uint32_t tS = tmem + Lay::cS, tdP = tmem + Lay::cdP;
      wait(br.held_full, 0);
      for (int t = 0; t < nt; ++t) {
        const int s = t % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(&br.full[s], (t / NS) & 1);
        if (t > 0) wait(br.consumed, (t - 1) & 1);
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tS, tc::desc_add(dKk, tc::kmajor_off(BW, kk)), tc::desc_add(dQk, so + tc::kmajor_off(BW, kk)),
                        idS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss_e(tdP, tc::desc_add(dVk, tc::kmajor_off(BW, kk)), tc::desc_add(ddOk, so + tc::kmajor_off(BW, kk)),
                        idS, kk > 0);
        ptx::mma_commit_e(br.s_full);
      }
    }
  } else if (warp == kCW + 2) {
    // -------------------------------------------------------- output MMAs
    if (ok) {
      constexpr uint32_t idKV = ptx::idesc_bf16(BW, D, 0, 1);  // A K-major (TMEM / dS^T), B MN-major
      constexpr uint32_t idQ = ptx::idesc_bf16(BW, D, 1, 1);   // A = dS read M-major, B = K MN-major
      const uint32_t sSt = ptx::smem_u32(sm + Lay::oStage), sdS = ptx::smem_u32(sm + Lay::odS);
      const uint64_t dQm = tc::mnmajor_desc(sSt, BW, 0), ddOm = tc::mnmajor_desc(sSt + kTile, BW, 0);
      const uint64_t dSk = tc::kmajor_desc(sdS, BW, 0);   // dS^T: M = keys, K = queries (2 slabs)
      const uint64_t dSm = tc::mnmajor_desc(sdS, BW, 0);  // dS: M = queries (2 slabs), K = keys
      const uint64_t dKm = tc::mnmajor_desc(ptx::smem_u32(sm + Lay::oK), BW, 0);  // K: K = keys, N = d
      const uint32_t tP = tmem + Lay::cP, tdV = tmem + Lay::cdV, tdK = tmem + Lay::cdK, tdQ = tmem + Lay::cdQ;
      for (int t = 0; t < nt; ++t) {
        const int s = t % NS;
        const uint32_t so = static_cast<uint32_t>(s * Lay::kStage);
        wait(br.ready, t & 1);
        // Already complete (the stage is refilled only after this block's products): the
        // acquire of the TMA-written stage for this warp's reads of Q_i and dO_i.
        wait(&br.full[s], (t / NS) & 1);
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < BW / 16; ++k) {
          const uint32_t acc = (t > 0 || k > 0) ? 1u : 0u;
          ptx::mma_ts_e(tdV, tP + k * 8, tc::desc_add(ddOm, so + 2048 * k), idKV, acc);
          ptx::mma_ss_e(tdK, tc::desc_add(dSk, tc::kmajor_off(BW, k)), tc::desc_add(dQm, so + 2048 * k), idKV, acc);
        }
        if (t > 0) {  // the previous block's dQ has left TMEM
          wait(br.dq_empty, (t - 1) & 1);
          ptx::tc_fence_after();
        }
#pragma unroll
        for (int k = 0; k < BW / 16; ++k)
          ptx::mma_ss_e(tdQ, tc::desc_add(dSm, 2048 * k), tc::desc_add(dKm, 2048 * k), idQ, k > 0 ? 1u : 0u);
        ptx::mma_commit_e(br.dq_full);
      }
      ptx::mma_commit_e(br.acc_full);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int qd = warp & 3, cg = warp >> 2;
    const int r = qd * 32 + lane;  // key row of the held block (TMEM lane) in the epilogue
    const uint32_t lo = static_cast<uint32_t>(qd * 32) << 16;
    const int key = kb * BW + r;
    const int c0 = cg * kC;
    // Score tiles are read with the 16-lane shapes: a thread sees 8 queries of its 32
    // (pairs 2(t%4) + 8k, k < 4) for 4 keys (rows t/4 + 8m of each 16-lane half), so the
    // statistics of its 4 query pairs are loaded once per block.
    const int g4 = lane >> 2, q4 = lane & 3;
    const uint64_t c2 = tc::pk2f(c, c);
    // last query each of this thread's four keys (rows g4 + 16 h + 8 m of its quarter) sees
    int khi[2][2] = {{0, 0}, {0, 0}};
    if constexpr (WIN) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < 2; ++m) khi[h][m] = bd.key_hi(kvh, kb * BW + qd * 32 + g4 + 16 * h + 8 * m);
    }
    // dQ_t out of TMEM (this thread: query 32 qd + lane, columns 16 cg ..) into the stage of
    // block t as two 128-byte-swizzled fp32 boxes of 32 columns (the TMA reduce's layout).
    // Called once dq_full of block t has been waited for (its products read nothing more).
    auto drain = [&](int t) {
      uint32_t qv[16];
      ptx::tmem_ld16(tmem + Lay::cdQ + static_cast<uint32_t>(cg * 16) + lo, qv);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(br.dq_empty);
      uint8_t* box = sm + Lay::oStage + (t % NS) * Lay::kStage + (cg >> 1) * kTile;
      const int q = qd * 32 + lane;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4*>(box + sw128(q, (cg & 1) * 4 + u)) =
            make_uint4(qv[4 * u], qv[4 * u + 1], qv[4 * u + 2], qv[4 * u + 3]);
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(&br.stg_full[t % NS]);
    };
    for (int t = 0; t < nt; ++t) {
      const int s = t % NS;
      int bhq, i;
      tile_at(t, bhq, i);
      (void)bhq;
      wait(br.s_full, t & 1);
      ptx::tc_fence_after();
      uint32_t sv[2][16], pv[2][16];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t la = lo + (static_cast<uint32_t>(16 * h) << 16);
        ptx::tmem_ld16x256_x4(tmem + Lay::cS + c0 + la, sv[h]);
        ptx::tmem_ld16x256_x4(tmem + Lay::cdP + c0 + la, pv[h]);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(br.consumed);
      // Statistics of the block's queries, pair-interleaved and negated:
      // float4 2m = (-L2, -L2', -D, -D') of queries 2m, 2m+1.
      const float4* st = reinterpret_cast<const float4*>(sm + Lay::oStage + s * Lay::kStage + 2 * kTile) + c0;
      float4 A[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) A[k] = st[8 * k + 2 * q4];
      const int qbase = i * BW + c0 + 2 * q4;    // query of column (k = 0, col 0)
      const int kbase = kb * BW + qd * 32 + g4;  // key of (h = 0, row 0)
      uint32_t pk[2][8], dk[2][8];               // [h][2k + (row, row+8)]
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
      if ((causal && i == kb) || (WIN && causal && i * BW + BW - 1 > hi_first) || i * BW + c0 + kC > N)
        block(std::true_type{});
      else
        block(std::false_type{});
      if (t > 0) {  // the previous block's three products have read P^T and dS
        wait(br.dq_full, (t - 1) & 1);
        ptx::tc_fence_after();
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t la = lo + (static_cast<uint32_t>(16 * h) << 16);
        ptx::tmem_st16x128_x4(tmem + Lay::cP + c0 / 2 + la, pk[h]);
      }
      // dS into shared memory (key rows, 128-byte lines of queries): the thread's values
      // are the fragments of 8x8 matrices (rows: keys 8m + g4 of half h, columns: the 8
      // queries of chunk k), so one stmatrix writes the four chunks k of a (h, m); the
      // thread gives the address of row lane % 8 of chunk lane / 8.
      {
        const uint32_t sdS = ptx::smem_u32(sm + Lay::odS);
        const int qcol = c0 + 8 * (lane >> 3);  // first query of the chunk this lane addresses
        const uint32_t cbase = sdS + static_cast<uint32_t>((qcol >> 6) * kTile);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int kr = qd * 32 + 16 * h + 8 * m + (lane & 7);
            ptx::stmatrix_x4(cbase + sw128(kr, (qcol & 63) >> 3), dk[h][m], dk[h][2 + m], dk[h][4 + m], dk[h][6 + m]);
          }
      }
      ptx::fence_proxy_async_smem();
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(br.ready);
      // Block t-1's dQ leaves TMEM while this block's dV and dK products run (the output
      // warp starts dQ_t only after dq_empty).
      if (t > 0) drain(t - 1);
    }
    if (nt > 0) {
      wait(br.dq_full, (nt - 1) & 1);
      ptx::tc_fence_after();
      drain(nt - 1);
    }
    wait(br.acc_full, 0);
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

// D_i = dO_i . O_i and the row statistics the key-block pass reads, pair-interleaved and
// negated as the row passes write them: float4 2m = (-L2m log2 e, -L2m+1 log2 e, -D2m,
// -D2m+1), float4 2m+1 = 0 (no GProj coefficient); the padding row of an odd-length slice
// gets zeros.  The rows of the dQ accumulator are zeroed.  Eight threads per row, each
// with eight of the head dim's columns.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       const float* __restrict__ lse, float* __restrict__ stats,
                                                       float* __restrict__ acc, int64_t N, int64_t Np, int64_t BH,
                                                       int dv) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rowg = gid >> 3;  // (slice, row) over Np rows per slice
  const int part = static_cast<int>(gid & 7);
  const bool valid = rowg < BH * Np;  // every lane stays for the shuffles below
  const int64_t bh = valid ? rowg / Np : 0, row = valid ? rowg - bh * Np : 0;
  const bool live = valid && row < N;
  float dsum = 0.f;
  if (live) {
    const int64_t off = (bh * N + row) * dv + part * 8;
    if (part * 8 < dv) {
      const uint4 a = *reinterpret_cast<const uint4*>(O + off);
      const uint4 b = *reinterpret_cast<const uint4*>(dO + off);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dsum += tc::bf16_lo(aw[e]) * tc::bf16_lo(bw[e]) + tc::bf16_hi(aw[e]) * tc::bf16_hi(bw[e]);
    }
    float4* ar = reinterpret_cast<float4*>(acc + (bh * N + row) * 64 + part * 8);
    ar[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    ar[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
  dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
  dsum += __shfl_xor_sync(0xffffffffu, dsum, 4);
  if (valid && part == 0) {
    float* wf = stats + bh * Np * 4;
    const int64_t k2 = row & ~static_cast<int64_t>(1);
    const int odd = static_cast<int>(row & 1);
    wf[k2 * 4 + odd] = live ? -lse[bh * N + row] * kLog2e : 0.f;
    wf[k2 * 4 + 2 + odd] = live ? -dsum : 0.f;
    wf[(k2 + 1) * 4 + odd] = 0.f;
    wf[(k2 + 1) * 4 + 2 + odd] = 0.f;
  }
}

// dQ = bf16(s acc), the head dim's dv columns of each row, eight per thread.
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dQ,
                                                     int64_t rows, int dv, float scale) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gid >> 3;
  const int part = static_cast<int>(gid & 7);
  if (row >= rows || part * 8 >= dv) return;
  const float4* a = reinterpret_cast<const float4*>(acc + row * 64 + part * 8);
  const float4 x = a[0], y = a[1];
  *reinterpret_cast<uint4*>(dQ + row * dv + part * 8) =
      make_uint4(ptx::pack_bf16(scale * x.x, scale * x.y), ptx::pack_bf16(scale * x.z, scale * x.w),
                 ptx::pack_bf16(scale * y.x, scale * y.y), ptx::pack_bf16(scale * y.z, scale * y.w));
}

}  // namespace

bool bwd_fused_applies(const Problem& p, bool gproj) { return bwd_single_pass(p.dtype, p.d, p.N, gproj); }

cudaError_t tc_bwd_fused(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* lse, void* dQ, void* dK, void* dV, float4* ws,
                         cudaStream_t st) {
  if (p.d > D) return cudaErrorInvalidValue;
  const int64_t N = p.N, BH = p.BH, Np = (p.N + 1) & ~static_cast<int64_t>(1), d = p.d;
  float* stats = reinterpret_cast<float*>(ws);
  float* acc = reinterpret_cast<float*>(ws + BH * Np);  // behind the statistics (16 bytes per row)
  alignas(64) CUtensorMap q, g, k, v, s, a;
  // Tensor maps over the true head dim d <= D: TMA zero-fills the padding columns.
  if (!make_tmap_bf16(&q, Q, N, d, BH, BW) || !make_tmap_bf16(&g, dO, N, d, BH, BW) ||
      !make_tmap_bf16(&k, K, N, d, p.BHkv, BW) || !make_tmap_bf16(&v, V, N, d, p.BHkv, BW) ||
      !make_tmap_stats(&s, stats, Np, BH, BW) || !make_tmap_f32_rows(&a, acc, N, BH, BW))
    return cudaErrorInvalidValue;
  const int64_t prep_threads = BH * Np * 8;
  bwd_prep_kernel<<<static_cast<unsigned>((prep_threads + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), lse, stats, acc, N, Np, BH,
      static_cast<int>(d));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nb = static_cast<int>((N + BW - 1) / BW);
  auto kern = banded(p) ? bwd_fused_kernel<true, true>
              : p.group > 1 ? bwd_fused_kernel<true, false>
                            : bwd_fused_kernel<false, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::bytes);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(nb * p.BHkv), kThreads, Lay::bytes, st>>>(
      k, v, q, g, s, a, static_cast<__nv_bfloat16*>(dK), static_cast<__nv_bfloat16*>(dV), static_cast<int>(N), nb,
      static_cast<int>(p.BHkv), p.scale, p.scale * kLog2e, p.causal, make_band(p, eff_window_tc(p), true), p.group,
      static_cast<int>(d));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t cv_threads = BH * N * 8;
  bwd_dq_kernel<<<static_cast<unsigned>((cv_threads + 255) / 256), 256, 0, st>>>(
      acc, static_cast<__nv_bfloat16*>(dQ), BH * N, static_cast<int>(d), p.scale);
  return cudaGetLastError();
}

uint32_t tc_bwd_fused_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
