// Internal launch interface between the C ABI (api.cu) and the kernel
// translation units.  Every launcher validates nothing: api.cu has already
// checked pointers, sizes, alignment and workspace.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "fbd.h"

namespace fbd {

struct Problem {
  int64_t B, H, N, d;
  int64_t BH;     // B * H independent (batch, head) slices
  float scale;    // s, already resolved (1/sqrt(d) when the caller passed 0)
  int dtype;      // attn_dtype_t
  int causal;     // 1: key j visible to query i iff j <= i; 0: every key visible
  int group;      // query heads per key/value head (1: multi-head attention)
  int64_t BHkv;   // B * H / group key/value slices; query slice bh reads slice bh / group
  int64_t window; // causal sliding window W (key j visible to row i iff i - W < j <= i), 1 <= W < N;
                  // 0: none (also when the caller's W >= N, which is the plain causal mask)
  const int* seg_lo;  // document mask: first key of each row's document, [B][N] (nullptr: none)
  const int* seg_hi;  // ... last row of each key's document, [B][N]
};

// A banded causal mask is in force: the window, the document bounds, or both.
inline bool banded(const Problem& p) { return p.window > 0 || p.seg_lo != nullptr; }

// The banded causal mask as the kernels take it (by value): row i sees the keys
// lo(i) <= j <= i and key j is seen by the rows j <= i <= hi(j), with
// lo(i) = max(i - W + 1, seg_lo[i], 0) and hi(j) = min(j + W - 1, seg_hi[j], N - 1), each
// term only where given.  A slice index s (query slice in row passes, key/value slice in
// column passes) belongs to batch row s / hpb.  Positions past N are looked up at N - 1.
struct Band {
  int64_t N;
  int64_t win;   // W, or larger than N plus a block when there is no window
  int64_t hpb;   // slices per batch row of the slice index the kernel holds
  const int* lo;
  const int* hi;
  __device__ __forceinline__ int row_lo(int64_t slice, int64_t i) const {
    int64_t l = i - win + 1;
    if (lo != nullptr) {
      const int64_t v = lo[(slice / hpb) * N + (i < N ? i : N - 1)];
      l = l > v ? l : v;
    }
    return static_cast<int>(l > 0 ? l : 0);
  }
  __device__ __forceinline__ int key_hi(int64_t slice, int64_t j) const {
    int64_t h = j + win - 1;
    if (hi != nullptr) {
      const int64_t v = hi[(slice / hpb) * N + (j < N ? j : N - 1)];
      h = h < v ? h : v;
    }
    return static_cast<int>(h < N - 1 ? h : N - 1);
  }
};
inline Band make_band(const Problem& p, int64_t win, bool kv_slices) {
  return Band{p.N, win, kv_slices ? p.BHkv / p.B : p.H, p.seg_lo, p.seg_hi};
}

// The window as the kernels take it: W, or N + 1 when there is none (then i - W + 1 <= 0
// and j + W > N for every row i and key j, so the window bounds never bind).
inline int64_t eff_window(const Problem& p) { return p.window > 0 ? p.window : p.N + 1; }
// The same for the tensor-core kernels (int): with no window, larger than N plus one
// block of 256 rows, so that no block bound derived from it ever binds.
inline int64_t eff_window_tc(const Problem& p) { return p.window > 0 ? p.window : p.N + 512; }

// CUDA-core kernel (simt.cu): the GProj projected-dS diagnostic export (bf16 inputs).
cudaError_t simt_projected_dS(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* lse, float* dS, cudaStream_t st);

// Document bounds from segment ids (mask.cu): lo[b][i] = first index of i's run of equal
// ids, hi[b][j] = last index of j's run (binary searches; ids non-decreasing along N).
cudaError_t segment_bounds(int64_t B, int64_t N, const int* seg, int* lo, int* hi, cudaStream_t st);

// The tf32 tensor-core engine (tc_f32.cu): kind::tf32 MMAs, each product as three tf32
// products of the operands' high and low parts, synchronous steps.  It serves float32
// inputs at every head dim (tc32_supports; GProj does not apply to float32) and the bf16
// case that has no bf16 kernel: the BoB (with or without GProj) at d = 256, with the GProj
// rounding of dS and P applied in fp32.  Workspace layout: one
// float4 of row statistics or states per row at slice pitch N; GProj BoB coefficients
// one float per row at pitch N in bob_rho_region.
bool tc32_supports(int64_t d);
cudaError_t tc32_fwd(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse,
                     cudaStream_t st);
cudaError_t tc32_bwd(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes, cudaStream_t st);
cudaError_t tc32_bob(const Problem& p, const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* lse, const void* a, const void* b, const void* c, void* gQ, void* gK, void* gV,
                     void* gdO, bool gproj, float4* ws, int passes, cudaStream_t st);
uint32_t tc32_take_error();

// bf16 tensor-core path (tcgen05 + TMA).  Return cudaErrorInvalidValue if a
// tensor map could not be encoded.
cudaError_t tc_fwd(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* lse,
                   cudaStream_t st);
cudaError_t tc_bwd(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* lse, void* dQ, void* dK, void* dV, int gproj, float4* ws,
                   int passes, cudaStream_t st);
// The 128-wide backward kernels (tc_bwd_wide.cu): both passes at d <= 64, with or
// without GProj; the row pass alone at 64 < d <= 128 without GProj.
cudaError_t tc_bwd_wide(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* lse, void* dQ, void* dK, void* dV, float4* ws, int passes,
                        cudaStream_t st, bool gproj = false);
// Single-pass backward (tc_bwd_fused.cu), bf16 at d <= 64 without GProj: a prep launch
// (D_i, the row statistics, a zeroed fp32 dQ accumulator), one launch per key block that
// writes dK, dV once and reduce-adds each query block's dS K into the accumulator, and a
// launch that scales and rounds dQ.  `ws` holds the statistics (16 bytes per row, rows of
// a slice rounded up to even) and then the accumulator (bwd_fused_acc_bytes).
//
// From N = 2^21 on the two-pass form is used instead: its reduce-adds of dQ shares, one
// per (key block, query block) pair, then run at ~2.5 TB/s instead of ~3.6, and the
// two passes (no reduction) are as fast at 2^21 and faster beyond (B1 H12 d64: 1165 vs
// 946 TFLOP/s at 2^20, 878 vs 888 at 2^21, 795 vs 876 at 2^22).
constexpr int64_t kBwdSinglePassMaxN = (int64_t{1} << 21) - 1;
inline bool bwd_single_pass(int dtype, int64_t d, int64_t N, bool gproj) {
  return dtype == ATTN_BF16 && d > 0 && d <= 64 && !gproj && N <= kBwdSinglePassMaxN;
}
bool bwd_fused_applies(const Problem& p, bool gproj);
inline size_t bwd_fused_acc_bytes(int64_t BH, int64_t N) { return static_cast<size_t>(BH) * N * 64 * sizeof(float); }
cudaError_t tc_bwd_fused(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* lse, void* dQ, void* dK, void* dV, float4* ws, cudaStream_t st);
uint32_t tc_bwd_fused_take_error();

cudaError_t tc_bob(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* lse, const void* a, const void* b, const void* c, void* gQ,
                   void* gK, void* gV, void* gdO, bool gproj, float4* ws, int passes, cudaStream_t st);
// d = 128: the same passes with each block of rows (keys) split over two CTAs by
// output half (tc_bob128.cu).
cudaError_t tc_bob128(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                      const void* dO, const float* lse, const void* a, const void* b, const void* c, void* gQ,
                      void* gK, void* gV, void* gdO, bool gproj, float4* ws, int passes, cudaStream_t st);
// BoB with GProj, tensor-core path: Pb_i = sum_j P^_ij b_j (fp32, bob_pb_cols(d) per
// row) for every row, P^ = bf16(2^(S s log2 e - L log2 e)) formed exactly as the BoB row
// pass forms it (the forward kernel run with the stored L and b in place of V; tc_fwd.cu).
cudaError_t tc_bob_pb(const Problem& p, const void* Q, const void* K, const void* b, const float* lse, float* pb,
                      cudaStream_t st);

// BoB workspace: the row states (16 bytes per row, the rows of a slice rounded up to
// an even count); with GProj (bf16) a region of the same size for the GProj
// coefficients (one float per row: at pitch bob_rho_pitch(N) on the tensor-core path,
// at pitch N on the CUDA-core path), and on the tensor-core path the rows' P^ b (fp32,
// bob_pb_cols(d) per row, B*H*N rows).
inline int64_t bob_state_rows(const Problem& p) { return p.BH * ((p.N + 1) & ~static_cast<int64_t>(1)); }
inline float4* bob_rho_region(float4* ws, const Problem& p) { return ws + bob_state_rows(p); }
inline float* bob_pb_region(float4* ws, const Problem& p) {
  return reinterpret_cast<float*>(ws + 2 * bob_state_rows(p));
}
inline int bob_pb_cols(int64_t d) { return d <= 64 ? 64 : 128; }
// Tensor-core path: the coefficients are one float per row, -rho_i, the rows of a slice
// rounded up to a multiple of 4 (read by TMA as float4 groups).
__host__ __device__ inline int64_t bob_rho_pitch(int64_t N) { return (N + 3) & ~static_cast<int64_t>(3); }

// passes: bit 0 = the row pass, bit 1 = the column pass (ATTN_ROW_PASS / ATTN_COL_PASS).

// Which kernels exist for a given (op, dtype, d): false means ATTN_ERR_UNSUPPORTED.
bool tc_supports(int op, int64_t d);  // op: 0 fwd, 1 bwd, 2 bob

// Device status words (bit FBD_ERR_TIMEOUT), read-and-cleared per translation unit.
uint32_t tc_fwd_take_error();
uint32_t tc_bwd_take_error();
uint32_t tc_bwd_wide_take_error();
uint32_t tc_bob_take_error();
uint32_t tc_bob128_take_error();
uint32_t selftest_take_error();

// One CTA whose bounded wait on an mbarrier that nothing completes gives up after
// 20 ms (selftest.cu): the failure-detection path, exercised without a fault.
cudaError_t selftest_wait_timeout(cudaStream_t st);

// Record `msg` as the calling thread's attn_last_error() detail; returns s.
attn_status_t set_last_error(attn_status_t s, const char* msg);

// The descriptor checks every entry point makes (ATTN_OK or the status attn_bob would return).
attn_status_t validate_desc(const attn_desc_t* desc);

// Tensor maps: 3-D bf16 view (d, N, B*H) of a [B,H,N,d] tensor, box (64, rows, 1),
// 128-byte swizzle.  Returns false if the driver entry point is missing or the
// encode fails.
bool make_tmap_bf16(void* map_out /* CUtensorMap* */, const void* base, int64_t N, int64_t d, int64_t BH,
                    int box_rows);

// Tensor map of an fp32 [B*H, N, 64] row buffer: 3-D view (64, N, B*H), box (32, rows, 1)
// (128 bytes of a row), 128-byte swizzle; rows past N are never written by a store or reduce.
bool make_tmap_f32_rows(void* map_out, const void* base, int64_t N, int64_t BH, int box_rows);

// Tensor map of the float4 row-statistics workspace [B*H, N]: 3-D fp32 view
// (4, N, B*H), box (4, rows, 1), no swizzle; rows past N read as zero.
bool make_tmap_stats(void* map_out, const void* base, int64_t N, int64_t BH, int box_rows);

}  // namespace fbd
