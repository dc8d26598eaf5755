// C ABI of libfbd (declared in include/fbd.h): argument validation, dispatch to
// the float32 CUDA-core kernels or the bf16 tcgen05/TMA kernels, and status
// reporting.  No entry point allocates device memory or falls back to another
// implementation: an unsupported request is an error.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "fbd.h"
#include "internal.h"

namespace {

thread_local char g_last_error[256] = "";

attn_status_t fail(attn_status_t s, const char* fmt, const char* what = "") {
  std::snprintf(g_last_error, sizeof(g_last_error), fmt, what);
  return s;
}

struct Span {
  const char* name;
  uintptr_t lo, hi;  // [lo, hi)
};

bool overlap(const Span& a, const Span& b) { return a.lo < b.hi && b.lo < a.hi; }

// Shape/type checks shared by every entry point.  Fills `p` on success.
attn_status_t check_desc(const attn_desc_t* desc, fbd::Problem& p) {
  if (desc == nullptr) return fail(ATTN_ERR_INVALID_ARG, "desc is NULL%s");
  if (desc->B < 0 || desc->H < 0 || desc->N < 0 || desc->d <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "negative B/H/N or non-positive d%s");
  if (desc->causal != 0 && desc->causal != 1) return fail(ATTN_ERR_UNSUPPORTED, "causal must be 0 or 1%s");
  if (desc->group < 0) return fail(ATTN_ERR_INVALID_ARG, "group must be >= 0%s");
  const int64_t g = desc->group == 0 ? 1 : desc->group;
  if (desc->H % g != 0) return fail(ATTN_ERR_INVALID_ARG, "group must divide H%s");
  if (desc->window < 0) return fail(ATTN_ERR_INVALID_ARG, "window must be >= 0%s");
  if (desc->window > 0 && desc->causal != 1)
    return fail(ATTN_ERR_UNSUPPORTED, "a window needs the causal mask (causal = 1)%s");
  if ((desc->seg_lo == nullptr) != (desc->seg_hi == nullptr))
    return fail(ATTN_ERR_INVALID_ARG, "seg_lo and seg_hi must both be set or both be NULL%s");
  if (desc->seg_lo != nullptr && desc->causal != 1)
    return fail(ATTN_ERR_UNSUPPORTED, "a document mask needs the causal mask (causal = 1)%s");
  if (desc->d != 32 && desc->d != 64 && desc->d != 96 && desc->d != 128 && desc->d != 256)
    return fail(ATTN_ERR_UNSUPPORTED, "head dim must be 32, 64, 96, 128 or 256%s");
  if (desc->dtype != ATTN_F32 && desc->dtype != ATTN_BF16) return fail(ATTN_ERR_UNSUPPORTED, "unknown dtype%s");
  if (!std::isfinite(desc->scale) || desc->scale < 0.f)
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and >= 0 (0 selects 1/sqrt(d))%s");
  // Overflow guards: element counts of one tensor must fit comfortably in int64,
  // the sequence length in a TMA coordinate (int32), slices in a 1-D grid.
  const int64_t lim = int64_t(1) << 31;
  if (desc->N >= lim || desc->B >= lim || desc->H >= lim)
    return fail(ATTN_ERR_INVALID_ARG, "B, H and N must each be < 2^31%s");
  const long double elems = (long double)desc->B * desc->H * desc->N * desc->d;
  if (elems > 9.0e18L / 8) return fail(ATTN_ERR_INVALID_ARG, "tensor too large%s");
  p.B = desc->B;
  p.H = desc->H;
  p.N = desc->N;
  p.d = desc->d;
  p.BH = desc->B * desc->H;
  p.scale = desc->scale == 0.f ? 1.0f / std::sqrt(static_cast<float>(desc->d)) : desc->scale;
  p.dtype = desc->dtype;
  p.causal = desc->causal;
  p.group = static_cast<int>(g);
  p.BHkv = p.BH / g;
  p.window = desc->window > 0 && desc->window < desc->N ? desc->window : 0;  // W >= N: the causal mask
  p.seg_lo = desc->seg_lo;
  p.seg_hi = desc->seg_hi;
  if (p.BH >= lim) return fail(ATTN_ERR_INVALID_ARG, "B*H must be < 2^31%s");
  if (((p.N + 7) / 8) * p.BH >= lim) return fail(ATTN_ERR_INVALID_ARG, "B*H*N too large for one launch%s");
  return ATTN_OK;
}

size_t elem_size(const fbd::Problem& p) { return p.dtype == ATTN_F32 ? 4 : 2; }

// Bytes of one [B, H / group, N, d] key/value-side tensor.
size_t kv_bytes(const fbd::Problem& p) { return static_cast<size_t>(p.BHkv * p.N * p.d) * elem_size(p); }

// Non-NULL, 16-byte aligned, pairwise non-overlapping outputs vs everything.
attn_status_t check_ptrs(const Span* in, int nin, const Span* out, int nout) {
  for (int k = 0; k < nin + nout; ++k) {
    const Span& s = k < nin ? in[k] : out[k - nin];
    if (s.lo == 0) return fail(ATTN_ERR_INVALID_ARG, "pointer %s is NULL", s.name);
    if (s.lo % 16 != 0) return fail(ATTN_ERR_ALIGNMENT, "pointer %s is not 16-byte aligned", s.name);
  }
  for (int k = 0; k < nout; ++k) {
    for (int m = 0; m < nin; ++m)
      if (overlap(out[k], in[m])) return fail(ATTN_ERR_INVALID_ARG, "output %s overlaps an input", out[k].name);
    for (int m = k + 1; m < nout; ++m)
      if (overlap(out[k], out[m])) return fail(ATTN_ERR_INVALID_ARG, "output %s overlaps another output", out[k].name);
  }
  return ATTN_OK;
}

Span span(const char* name, const void* ptr, size_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
  return Span{name, lo, lo + bytes};
}

// The inputs of an entry point, with the document bounds appended when they are given.
struct Inputs {
  Span s[13];
  int n = 0;
  Inputs(std::initializer_list<Span> l, const fbd::Problem& p) {
    for (const Span& x : l) s[n++] = x;
    if (p.seg_lo != nullptr) {
      const size_t b = static_cast<size_t>(p.B * p.N) * sizeof(int);
      s[n++] = span("seg_lo", p.seg_lo, b);
      s[n++] = span("seg_hi", p.seg_hi, b);
    }
  }
};

attn_status_t launch_status(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  (void)cudaGetLastError();  // clear the sticky-free launch error
  return fail(ATTN_ERR_LAUNCH, "CUDA: %s", cudaGetErrorString(e));
}

bool tc_path(const fbd::Problem& p, int op) { return p.dtype == ATTN_BF16 && fbd::tc_supports(op, p.d); }
// float32 inputs on the tensor cores (three tf32 products per product), every supported d.
bool tc32_path(const fbd::Problem& p) { return p.dtype == ATTN_F32 && fbd::tc32_supports(p.d); }

}  // namespace

namespace fbd {
// bf16 tensor-core kernels by operation: forward, backward and backward-over-backward
// for d in {64, 128}, and for d = 32 and 96 on those kernels with the head dim
// zero-padded to 64 and 128 in shared memory (TMA fills the columns past d with
// zeros, which add nothing to any product; nothing past d is stored).  BoB at
// d > 64 splits each block over two CTAs by output half: its row pass's four d-wide
// accumulators would otherwise fill the 512 TMEM columns.  At d = 256 the forward
// runs on tensor cores (64-key blocks, O in 256 TMEM columns), and so does the backward
// with and without GProj (one stage of streamed tiles; the column pass, and with GProj the
// row pass, split over two CTAs by output half); the BoB at d = 256 runs on the tf32
// tensor-core engine (tc_f32.cu, output columns in parts of 64 or 32): its d-wide
// accumulators and held operands do not fit beside the pipelined kernels' tiles.
bool tc_supports(int op, int64_t d) {
  if (d == 256) return op == 0 || op == 1;
  return d == 32 || d == 64 || d == 96 || d == 128;
}
}  // namespace fbd

namespace fbd {
attn_status_t set_last_error(attn_status_t s, const char* msg) { return fail(s, "%s", msg); }
attn_status_t validate_desc(const attn_desc_t* desc) {
  Problem p;
  return check_desc(desc, p);
}
}  // namespace fbd

extern "C" {

attn_status_t attn_fwd(const attn_desc_t* desc, const void* Q, const void* K, const void* V, void* O, float* lse,
                       void* stream) {
  fbd::Problem p;
  attn_status_t s = check_desc(desc, p);
  if (s != ATTN_OK) return s;
  if (p.BH * p.N == 0) return ATTN_OK;
  const size_t tb = static_cast<size_t>(p.BH * p.N * p.d) * elem_size(p), sb = p.BH * p.N * sizeof(float);
  const size_t kb = kv_bytes(p);
  const Inputs in({span("Q", Q, tb), span("K", K, kb), span("V", V, kb)}, p);
  const Span out[] = {span("O", O, tb), span("lse", lse, sb)};
  if ((s = check_ptrs(in.s, in.n, out, 2)) != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (tc32_path(p)) return launch_status(fbd::tc32_fwd(p, Q, K, V, O, lse, st));
  return launch_status(fbd::tc_fwd(p, Q, K, V, O, lse, st));  // bf16: tensor cores at every d
}

size_t attn_bwd_workspace_bytes(const attn_desc_t* desc, int gproj) {
  if (desc == nullptr || desc->B < 0 || desc->H < 0 || desc->N < 0) return 0;
  // 16 bytes per row, the rows of each slice rounded up to an even count (the bf16
  // column pass reads the row statistics two rows at a time); for the single-pass bf16
  // backward (d <= 64, no GProj, N < 2^21) then the fp32 dQ accumulator, 256 bytes per row.
  size_t n = static_cast<size_t>(desc->B) * desc->H * ((desc->N + 1) & ~static_cast<int64_t>(1)) * 16;
  if (fbd::bwd_single_pass(desc->dtype, desc->d, desc->N, gproj != 0))
    n += fbd::bwd_fused_acc_bytes(desc->B * desc->H, desc->N);
  return n;
}

size_t attn_bob_workspace_bytes(const attn_desc_t* desc, int gproj) {
  if (desc == nullptr || desc->B < 0 || desc->H < 0 || desc->N < 0) return 0;
  // The row states: 16 bytes per row, rows of each slice rounded up to an even count
  // (the bf16 column pass reads them two rows at a time).  GProj (bf16 only): as much
  // again for the coefficients, and on the tensor-core path (d <= 128) the rows' P^ b
  // in fp32 (64 or 128 per row).  The layout is fbd::bob_rho_region / bob_pb_region.
  const size_t rows = static_cast<size_t>(desc->B) * desc->H * ((desc->N + 1) & ~static_cast<int64_t>(1));
  size_t n = rows * 16;
  if (gproj && desc->dtype == ATTN_BF16) {
    n += rows * 16;
    if (desc->d <= 128)
      n += static_cast<size_t>(desc->B) * desc->H * desc->N * fbd::bob_pb_cols(desc->d) * sizeof(float);
  }
  return n;
}

attn_status_t attn_bwd_passes(const attn_desc_t* desc, const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* lse, void* dQ, void* dK, void* dV, int gproj,
                              void* workspace, size_t workspace_bytes, int passes, void* stream) {
  fbd::Problem p;
  attn_status_t s = check_desc(desc, p);
  if (s != ATTN_OK) return s;
  if (passes < 1 || passes > 3) return fail(ATTN_ERR_INVALID_ARG, "passes must be ATTN_ROW_PASS, ATTN_COL_PASS or both%s");
  if (p.BH * p.N == 0) return ATTN_OK;
  // One pass alone reads or writes only the row statistics (the first 16 bytes per row of
  // the workspace); both passes in one call may take the single-pass form's accumulator.
  const size_t stats_bytes = static_cast<size_t>(p.BH) * ((p.N + 1) & ~static_cast<int64_t>(1)) * 16;
  const size_t need = passes == (ATTN_ROW_PASS | ATTN_COL_PASS) ? attn_bwd_workspace_bytes(desc, gproj) : stats_bytes;
  if (workspace == nullptr || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace NULL or smaller than attn_bwd_workspace_bytes()%s");
  const size_t tb = static_cast<size_t>(p.BH * p.N * p.d) * elem_size(p), sb = p.BH * p.N * sizeof(float);
  const size_t kb = kv_bytes(p);
  const Inputs in({span("Q", Q, tb), span("K", K, kb), span("V", V, kb), span("O", O, tb), span("dO", dO, tb),
                   span("lse", lse, sb)}, p);
  const Span out[] = {span("dQ", dQ, tb), span("dK", dK, kb), span("dV", dV, kb),
                      span("workspace", workspace, need)};
  if ((s = check_ptrs(in.s, in.n, out, 4)) != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float4* ws = static_cast<float4*>(workspace);
  // float32 at every d: the tf32 engine (GProj does not apply).
  if (tc32_path(p)) return launch_status(fbd::tc32_bwd(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, passes, st));
  // Both passes in one call: the single-pass form where it exists (bf16, d <= 64, no GProj).
  if (passes == (ATTN_ROW_PASS | ATTN_COL_PASS) && fbd::bwd_fused_applies(p, gproj != 0))
    return launch_status(fbd::tc_bwd_fused(p, Q, K, V, O, dO, lse, dQ, dK, dV, ws, st));
  return launch_status(fbd::tc_bwd(p, Q, K, V, O, dO, lse, dQ, dK, dV, gproj != 0, ws, passes, st));
}

attn_status_t attn_bwd(const attn_desc_t* desc, const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* lse, void* dQ, void* dK, void* dV, int gproj, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return attn_bwd_passes(desc, Q, K, V, O, dO, lse, dQ, dK, dV, gproj, workspace, workspace_bytes,
                         ATTN_ROW_PASS | ATTN_COL_PASS, stream);
}

attn_status_t attn_bob_passes(const attn_desc_t* desc, const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* lse, const void* gdQ, const void* gdK, const void* gdV,
                              void* gQ, void* gK, void* gV, void* gdO, int gproj, void* workspace,
                              size_t workspace_bytes, int passes, void* stream) {
  fbd::Problem p;
  attn_status_t s = check_desc(desc, p);
  if (s != ATTN_OK) return s;
  if (passes < 1 || passes > 3) return fail(ATTN_ERR_INVALID_ARG, "passes must be ATTN_ROW_PASS, ATTN_COL_PASS or both%s");
  if (p.BH * p.N == 0) return ATTN_OK;
  const bool gp = gproj != 0 && p.dtype == ATTN_BF16;  // float32 dS is never rounded
  const size_t need = attn_bob_workspace_bytes(desc, gproj);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace NULL or smaller than attn_bob_workspace_bytes()%s");
  const size_t tb = static_cast<size_t>(p.BH * p.N * p.d) * elem_size(p), sb = p.BH * p.N * sizeof(float);
  const size_t kb = kv_bytes(p);
  const Inputs in({span("Q", Q, tb), span("K", K, kb), span("V", V, kb), span("O", O, tb), span("dO", dO, tb),
                   span("lse", lse, sb), span("gdQ", gdQ, tb), span("gdK", gdK, kb), span("gdV", gdV, kb)}, p);
  const Span out[] = {span("gQ", gQ, tb), span("gK", gK, kb), span("gV", gV, kb), span("gdO", gdO, tb),
                      span("workspace", workspace, need)};
  if ((s = check_ptrs(in.s, in.n, out, 5)) != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float4* ws = static_cast<float4*>(workspace);
  // float32 at every d, and bf16 BoB past the bf16 BoB kernels (d = 256): the tf32 engine.
  if (tc32_path(p) || !tc_path(p, 2))
    return launch_status(fbd::tc32_bob(p, Q, K, V, O, dO, lse, gdQ, gdK, gdV, gQ, gK, gV, gdO, gp, ws, passes, st));
  if (p.d > 64)
    return launch_status(
        fbd::tc_bob128(p, Q, K, V, O, dO, lse, gdQ, gdK, gdV, gQ, gK, gV, gdO, gp, ws, passes, st));
  return launch_status(fbd::tc_bob(p, Q, K, V, O, dO, lse, gdQ, gdK, gdV, gQ, gK, gV, gdO, gp, ws, passes, st));
}

attn_status_t attn_bob(const attn_desc_t* desc, const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* lse, const void* gdQ, const void* gdK, const void* gdV,
                       void* gQ, void* gK, void* gV, void* gdO, int gproj, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return attn_bob_passes(desc, Q, K, V, O, dO, lse, gdQ, gdK, gdV, gQ, gK, gV, gdO, gproj, workspace,
                         workspace_bytes, ATTN_ROW_PASS | ATTN_COL_PASS, stream);
}

attn_status_t attn_bwd_projected_dS(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                                    const void* O, const void* dO, const float* lse, float* dS_out,
                                    void* stream) {
  fbd::Problem p;
  attn_status_t s = check_desc(desc, p);
  if (s != ATTN_OK) return s;
  if (p.dtype != ATTN_BF16) return fail(ATTN_ERR_UNSUPPORTED, "the GProj projection applies to bf16 only%s");
  if (p.BH * p.N == 0) return ATTN_OK;
  const size_t tb = static_cast<size_t>(p.BH * p.N * p.d) * 2, sb = p.BH * p.N * sizeof(float);
  const size_t ob = static_cast<size_t>(p.BH) * p.N * p.N * sizeof(float);
  const size_t kb = static_cast<size_t>(p.BHkv * p.N * p.d) * 2;
  const Inputs in({span("Q", Q, tb), span("K", K, kb), span("V", V, kb), span("O", O, tb), span("dO", dO, tb),
                   span("lse", lse, sb)}, p);
  const Span out[] = {span("dS_out", dS_out, ob)};
  if ((s = check_ptrs(in.s, in.n, out, 1)) != ATTN_OK) return s;
  return launch_status(fbd::simt_projected_dS(p, Q, K, V, O, dO, lse, dS_out, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_segment_bounds(int64_t B, int64_t N, const int32_t* seg, int32_t* seg_lo, int32_t* seg_hi,
                                  void* stream) {
  if (B < 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "negative B or N%s");
  if (N >= (int64_t(1) << 31) || B >= (int64_t(1) << 31) || (B > 0 && N > (int64_t(1) << 40) / B))
    return fail(ATTN_ERR_INVALID_ARG, "B and N must each be < 2^31 and B*N < 2^40%s");
  if (B * N == 0) return ATTN_OK;
  const size_t b = static_cast<size_t>(B * N) * sizeof(int32_t);
  const Span in[] = {span("seg", seg, b)};
  const Span out[] = {span("seg_lo", seg_lo, b), span("seg_hi", seg_hi, b)};
  attn_status_t s = check_ptrs(in, 1, out, 2);
  if (s != ATTN_OK) return s;
  return launch_status(fbd::segment_bounds(B, N, seg, seg_lo, seg_hi, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "CUDA: %s", cudaGetErrorString(e));
  const uint32_t flags = fbd::tc_fwd_take_error() | fbd::tc_bwd_take_error() | fbd::tc_bwd_wide_take_error() | fbd::tc_bwd_fused_take_error() |
                         fbd::tc_bob_take_error() | fbd::tc_bob128_take_error() | fbd::tc32_take_error() |
                         fbd::selftest_take_error();
  if (flags != 0) return fail(ATTN_ERR_TIMEOUT, "a device-side bounded wait gave up%s");
  return ATTN_OK;
}

attn_status_t attn_check_wait_timeout(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = fbd::selftest_wait_timeout(st);
  if (e != cudaSuccess) return launch_status(e);
  return attn_device_status(stream);
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_LAUNCH: return "CUDA launch or tensor-map error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case ATTN_ERR_DEVICE: return "no usable CUDA device";
  }
  return "unknown status";
}

const char* attn_last_error(void) { return g_last_error; }

const char* attn_version(void) { return "libfbd 0.2 (sm_103a: tcgen05/TMA bf16 kernels, tcgen05 tf32x3 engine for float32 and the bf16 BoB at d = 256)"; }

}  // extern "C"

// ------------------------------------------------------------- tensor maps
namespace fbd {

namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &f, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  });
  return fn;
}
}  // namespace

bool make_tmap_bf16(void* map_out, const void* base, int64_t N, int64_t d, int64_t BH, int box_rows) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N * d) * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f32_rows(void* map_out, const void* base, int64_t N, int64_t BH, int box_rows) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {256u, static_cast<cuuint64_t>(N) * 256u};
  const cuuint32_t box[3] = {32u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_stats(void* map_out, const void* base, int64_t N, int64_t BH, int box_rows) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {4u, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {16u, static_cast<cuuint64_t>(N) * 16u};
  const cuuint32_t box[3] = {4u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fbd
