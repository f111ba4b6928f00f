// Shared device helpers for libquads (sm_103a).
//
// NVFP4 element/scale arithmetic follows the NVFP4 description of the TRACE
// digest ("NVFP4 与 E2M1 码本": global scale + per-16-block scale, round to
// nearest E2M1 level) with every step an IEEE float32 operation, so that codes
// and scale bytes are reproducible bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/quads.h"

namespace quads {

constexpr int kBlock = 16;            // elements per block scale
constexpr int kScoreChunk = QUADS_SCORE_CHUNK_ROWS;
constexpr float kE2M1Max = 6.0f;
constexpr float kE4M3Max = 448.0f;

// ----------------------------------------------------------------- host status
void set_detail(const char* fmt, ...);
quads_status_t fail(quads_status_t s, const char* fmt, ...);
quads_status_t check_launch(const char* what, int kernels_launched);
int num_sms();
quads_status_t select_check_args(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                 const int32_t* group_offsets, int32_t num_groups,
                                 const int32_t* group_counts, const uint8_t* scales, const float* tensor_scale,
                                 const float* score_partials, int32_t k, const int32_t* sel,
                                 const uint8_t* r_codes, const uint8_t* r_scales,
                                 const float* r_tensor_scale, size_t* need);

// ------------------------------------------------------------ debug checks
// Bounds-checked builds (-DQUADS_DEBUG): an access whose index comes from
// data or from tile arithmetic is guarded by QDBG(index in range); a failed
// guard latches its source line in this translation unit's debug word (read
// by quads_device_status) and the access is skipped.  Release builds compile
// the guards away.
#ifdef QUADS_DEBUG
static __device__ int g_debug_line;
static __device__ long long g_debug_value;
__device__ __forceinline__ bool quads_dbg(bool ok, int line, long long value) {
  if (!ok && atomicCAS(&g_debug_line, 0, line) == 0) g_debug_value = value;
  return ok;
}
#define QDBG(cond) quads_dbg((cond), __LINE__, 0)
#define QDBGV(cond, value) quads_dbg((cond), __LINE__, (long long)(value))
// Host side: read and clear this translation unit's debug word (and the
// value recorded with it).
[[maybe_unused]] static int take_debug_line(long long* value) {
  int v = 0, z = 0;
  long long val = 0, zz = 0;
  cudaMemcpyFromSymbol(&v, g_debug_line, sizeof(int));
  cudaMemcpyFromSymbol(&val, g_debug_value, sizeof(long long));
  cudaMemcpyToSymbol(g_debug_line, &z, sizeof(int));
  cudaMemcpyToSymbol(g_debug_value, &zz, sizeof(long long));
  *value = val;
  return v;
}
#else
#define QDBG(cond) true
#define QDBGV(cond, value) true
[[maybe_unused]] static int take_debug_line(long long* value) {
  *value = 0;
  return 0;
}
#endif

// ------------------------------------------------------------ scale layouts
// Byte offset of scale column c (a 16-element block) of row r in the
// tensor-core layout: 128-row x 4-column blocks of 512 bytes, row-block major.
__host__ __device__ __forceinline__ int64_t sf_tc_offset(int64_t r, int64_t c, int64_t ncols16) {
  return ((r >> 7) * (ncols16 >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}
__host__ __device__ __forceinline__ int64_t sf_offset(int layout, int64_t r, int64_t c,
                                                      int64_t ncols16) {
  return layout == QUADS_SCALES_TCGEN05 ? sf_tc_offset(r, c, ncols16) : r * ncols16 + c;
}
// Bytes of a TCGEN05-layout scale array for rows x cols elements.
__host__ __device__ __forceinline__ int64_t sf_tc_bytes(int64_t rows, int64_t cols) {
  return ((rows + 127) / 128) * 128 * (cols / 16);
}

// ------------------------------------------------------------ conversions
// E4M3 byte -> float through the hardware E4M3 -> f16 converter (every E4M3
// value, subnormals included, is exact in f16, and f16 -> f32 is exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h;
  asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(h)
      : "r"(b & 0xFFu));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// Non-negative float -> E4M3 byte, nearest/even, saturating at 448.
__device__ __forceinline__ uint32_t f32_to_e4m3_sat(float u) {
  u = fminf(u, kE4M3Max);
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(u));
  return r & 0xFFu;
}

// Eight floats -> eight E2M1 codes packed in 32 bits (element i in nibble i).
__device__ __forceinline__ uint32_t f32x8_to_e2m1(const float* v) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
        "f"(v[7]));
  return out;
}

// E2M1 code (4 bits) -> float value, from the format: 2 exponent bits (bias 1),
// 1 mantissa bit, subnormal 0.5 step.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float mag = e == 0 ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (c & 8u) ? -mag : mag;
}

// A pair of scaled values rounded to E2M1 (nearest even, saturating), and the
// codes' values back as floats: hardware conversions both ways (a is the low
// nibble of the pair).
__device__ __forceinline__ void e2m1_round_pair(float a, float b, float& qa, float& qb) {
  uint32_t h;
  asm("{\n\t.reg .b8 c;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c, %2, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, c;\n\t}"
      : "=r"(h)
      : "f"(a), "f"(b));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  qa = f.x;
  qb = f.y;
}

// Eight packed codes -> eight floats via the hardware E2M1 -> f16 converter.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t packed, float* out) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(packed));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 hh = *reinterpret_cast<__half2*>(&h[i]);
    float2 f = __half22float2(hh);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Tensor scale from the tensor's absolute maximum: fl(amax / 2688), 1 if 0.
__device__ __forceinline__ float tensor_scale_from_amax(float amax) {
  float s = __fdiv_rn(amax, kE2M1Max * kE4M3Max);
  return s == 0.0f ? 1.0f : s;
}

struct BlockScale {
  uint32_t byte;  // E4M3 scale byte
  float d;        // E4M3value * s_t
  float r;        // 1 / d (correctly rounded)
  bool zero;      // d == 0 or 1/d overflowed: all codes 0
};

// Block scale of a 16-block with absolute maximum m under tensor scale s_t.
__device__ __forceinline__ BlockScale block_scale(float m, float s_t) {
  BlockScale b;
  float u = __fdiv_rn(m, __fmul_rn(kE2M1Max, s_t));
  b.byte = f32_to_e4m3_sat(u);
  b.d = __fmul_rn(e4m3_to_f32(b.byte), s_t);
  b.r = __frcp_rn(b.d);
  b.zero = (b.d == 0.0f) || isinf(b.r);
  return b;
}

// Block scale for a byte that is already known (decode side).
__device__ __forceinline__ BlockScale block_scale_from_byte(uint32_t byte, float s_t) {
  BlockScale b;
  b.byte = byte;
  b.d = __fmul_rn(e4m3_to_f32(byte), s_t);
  b.r = __frcp_rn(b.d);
  b.zero = (b.d == 0.0f) || isinf(b.r);
  return b;
}

// MXFP4 block scale (OCP microscaling): 2^e with e = floor(log2 m) - 2 for the
// 32-block maximum m (2 = exponent of the largest E2M1 level), clamped at
// -127, stored as the E8M0 byte e + 127.  From the float's exponent field:
// floor(log2 m) = field - 127 for normal m; m below 2^-125 (field < 2) clamps.
__device__ __forceinline__ uint32_t e8m0_scale_byte(float m) {
  const uint32_t field = (__float_as_uint(m) >> 23) & 0xFFu;
  return field >= 2u ? field - 2u : 0u;
}
// 2^e and 2^-e of an E8M0 byte (e in [-127, 125] here: both are floats).
__device__ __forceinline__ float e8m0_value(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}
__device__ __forceinline__ float e8m0_inverse(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}

// Two float32 products per instruction (mul.rn.f32x2, sm_100+): each half is
// rounded as __fmul_rn rounds it.  Only for products that feed no addition:
// ptxas contracts an f32x2 multiply and a following f32x2 add or subtract into
// a fused multiply-add despite the .rn qualifiers (measured on the GB300:
// 16 % of residuals differed from the scalar two-rounding sequence), which
// the float32 orders fixed by the score and residual definitions forbid.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Quantize 8 values of one block: returns packed codes; writes levels*d residuals
// when want_residual.
__device__ __forceinline__ uint32_t quantize8(const float* x, const BlockScale& bs) {
  float v[8];
  const uint64_t rr = f2_pack(bs.r, bs.r);
#pragma unroll
  for (int i = 0; i < 8; i += 2) f2_unpack(f2_mul(f2_pack(x[i], x[i + 1]), rr), v[i], v[i + 1]);
  uint32_t c = f32x8_to_e2m1(v);
  return bs.zero ? 0u : c;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------ dependent launches
// The kernels of the layer path open with griddep_wait(): launched with
// programmatic stream serialization (launch_dep) a kernel may be scheduled
// while its stream predecessor still runs, and blocks there until that grid
// has completed and its memory writes are visible (launched plainly, the
// wait returns at once).  griddep_launch_dependents() then allows the
// stream's next kernel to be scheduled in turn, so its launch overlaps this
// kernel instead of following it.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... P, typename... A>
static inline cudaError_t launch_dep(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

// Group index of `row` for ascending offsets goff[0..G] (binary search).
__device__ __forceinline__ int group_of(const int32_t* goff, int G, int64_t row) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (goff[mid] <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace quads
