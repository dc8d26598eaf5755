// Helpers shared by the tcgen05 kernels: operand descriptors for TMA-written
// 128-byte-swizzled tiles, named barriers, bf16 packing.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fbd {
namespace tc {

// A tile of `rows` rows x D bf16 columns is stored as D/64 slabs; slab c holds
// columns [64c, 64c + 64) as `rows` lines of 128 bytes, 128-byte swizzled (the
// layout a TMA box of (64, rows) writes).  The tile base is 1024-byte aligned.

// K-major operand (rows = M or N index, columns = K), advanced to K-step k (16 columns).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int rows, int k) {
  return ptx::sdesc_sw128(base + (k >> 2) * rows * 128 + (k & 3) * 32, 16, 1024);
}
// Byte offset of K-step k within a K-major operand of `rows` rows (what kmajor_desc adds).
__host__ __device__ constexpr uint32_t kmajor_off(int rows, int k) {
  return static_cast<uint32_t>((k >> 2) * rows * 128 + (k & 3) * 32);
}
// MN-major operand (rows = K index, columns = M or N), advanced to K-step k (16 rows).
// Leading byte offset = slab stride (next 64 columns), stride byte offset = 8 rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int rows, int k) {
  return ptx::sdesc_sw128(base + k * 16 * 128, rows * 128, 1024);
}

// A descriptor moved by `bytes` within shared memory: the start address sits in
// bits 0-13 of the low word in 16-byte units, and every operand of these kernels
// lies in the first 256 KB, so the move never carries out of the low word.  The
// MMA warps build their descriptors once and step them with this single add, so
// the issuing thread spends few instructions per MMA (it shares its scheduler
// with two compute warps).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(d));
  lo += bytes >> 4;
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

// Barrier among the first `n` threads (the compute warps), id 1 (id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Grid order of the 1-D grids: slices (batch, head) go in groups of 8, so the
// streamed tiles of one group (K, V, ... of 8 heads) stay resident in L2 while its
// CTAs run; within a group, block index k = 0 (the heaviest causal block) comes
// first, interleaved across the group's slices.
struct Order {
  int bh, k;
};
__device__ __forceinline__ Order grid_order_at(int x, int BH, int nblk) {
  constexpr int G = 8;
  const int group = x / (G * nblk);
  const int base = group * G;
  const int gsize = min(G, BH - base);
  const int within = x - base * nblk;
  Order o;
  o.k = within / gsize;
  o.bh = base + within % gsize;
  return o;
}
__device__ __forceinline__ Order grid_order(int BH, int nblk) {
  return grid_order_at(static_cast<int>(blockIdx.x), BH, nblk);
}

// The two floats held by a packed bf16x2 word (low half = even element).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float f(uint32_t u) { return __uint_as_float(u); }

// Packed fp32 pairs (f32x2 arithmetic, two lanes per instruction).  A pair is a
// 64-bit register; element 0 in the low half.
__device__ __forceinline__ uint64_t pk2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ uint64_t pk2f(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpk2(uint64_t x) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// acc + the bf16 held in the low (high) half of w, in one mixed-precision add: the
// widening of a bf16 to fp32 is exact, so this rounds exactly as widening and then
// adding in fp32 would.
__device__ __forceinline__ float add_bf16_lo(float acc, uint32_t w) {
  float r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, l, %2;\n\t}" : "=f"(r) : "r"(w), "f"(acc));
  return r;
}
__device__ __forceinline__ float add_bf16_hi(float acc, uint32_t w) {
  float r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, h, %2;\n\t}" : "=f"(r) : "r"(w), "f"(acc));
  return r;
}

// The bf16x2 word as an fp32 pair (exact widening).
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) { return pk2(w << 16, w & 0xffff0000u); }

}  // namespace tc
}  // namespace fbd
