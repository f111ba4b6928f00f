// Activation-side kernels: tensor amax, NVFP4 RTN quantization with fused
// residual-energy partials (and the trainer's W4A16 fake quantization), top-k
// residual channel selection, the second quantization of the residual slice,
// TRACE rollout-guided rounding (full rollout codes or the 1-bit record), and
// the MXFP4 quantizer.
//
// [TRACE digest] "NVFP4 与 E2M1 码本": per-tensor scale + per-block scale, RTN.
// [QUADS technical summary] 2.1: Delta X_q = X - DQ(Q(X)); 2.2 A: asymmetric
// W4A16 QAT (weights fake-quantized on the trainer); 2.2 B "Mechanism":
// second-pass quantization of the channels with the largest FP4 error;
// "Implementation": a channel mask picks the top channels by residual magnitude.
// [TRACE digest] "核心方法", Eq. (3): q_TRACE = argmin_{q in {q-, q+}} |q - q_rollout|;
// the mantissa-only record; "技术新颖性": also validated on MXFP4.
//
// The streaming kernels read every byte once with 16-byte vector loads (8 bf16
// per lane) and take 16-element block maxima with warp shuffles; shared memory
// is used where values must be re-ordered: the residual squares summed per
// column in row order, and the top-k histograms.
#include <cstdio>

#include "common.cuh"

namespace quads {

static __device__ int g_quant_error;  // device-side argument check failures

constexpr int kRselGroupMin = 32;     // groups from which the per-group R_sel kernel is used
constexpr int kFusedMaxK = 1024;      // selected channels of the fused activation-side kernel
constexpr int kSmemGroups = 256;      // groups whose offsets and scales a quantizer block caches

// ---------------------------------------------------------------- amax
// One block per 8-row slice (inside one group), threads over (row, 8-col
// vector), eight 16-byte loads in flight per thread; the absolute maximum is
// taken on packed bf16 pairs (exact: the maximum of bf16 values is one of
// them) and converted to float once per thread.
constexpr int kAmaxRows = 8;
__global__ void __launch_bounds__(256) amax_kernel(const __nv_bfloat16* __restrict__ x,
                                                   int64_t rows, int cols, int64_t ldx,
                                                   const int32_t* __restrict__ row_index,
                                                   const int32_t* __restrict__ goff, int G,
                                                   uint32_t* __restrict__ amax_bits,
                                                   const int32_t* __restrict__ gcnt) {
  griddep_wait();
  const int64_t end = goff ? (int64_t)goff[G] : rows;
  const int vec_per_row = cols >> 3;
  const int64_t nslices = (end + kAmaxRows - 1) / kAmaxRows;
  __shared__ float red[8];
  for (int64_t slice = blockIdx.x; slice < nslices; slice += gridDim.x) {
    const int64_t r0 = slice * kAmaxRows;
    const int64_t r1 = min(r0 + kAmaxRows, end);
    const int g = goff ? group_of(goff, G, r0) : 0;
    if (goff && r1 > goff[g + 1]) atomicExch(&g_quant_error, QUADS_ERR_DEVICE_CHECK);
    __nv_bfloat162 m2 = __floats2bfloat162_rn(0.0f, 0.0f);
    // rows past the group's count (gcnt) are zero rows: not read
    const int64_t r1r = gcnt ? max(r0, min(r1, (int64_t)goff[g] + __ldg(gcnt + g))) : r1;
    const int total = (int)(r1r - r0) * vec_per_row;
    for (int i0 = threadIdx.x; i0 < total; i0 += 8 * blockDim.x) {
      uint4 u[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * blockDim.x;
        u[q] = make_uint4(0, 0, 0, 0);
        if (i < total) {
          const int rr = i / vec_per_row;
          const int64_t src = row_index ? (int64_t)row_index[r0 + rr] : r0 + rr;
          u[q] = __ldg(reinterpret_cast<const uint4*>(x + src * ldx) + (i - rr * vec_per_row));
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[j])));
      }
    }
    const float2 mf = __bfloat1622float2(m2);
    float m = fmaxf(mf.x, mf.y);
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
      float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
      v = warp_max(v);
      if (threadIdx.x == 0 && v > 0.0f) atomicMax(&amax_bits[g], __float_as_uint(v));
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- quantize
// A block owns one (32-row chunk, 256-column slab) task.  Warp w quantizes
// rows 4w .. 4w+3 of the chunk, two rows at a time: lane l takes the 16-element
// block (l & 15) of row (l >> 4), so each block scale is computed once.  In
// score mode every residual square R^2 is parked in shared memory and, after a
// barrier, thread c adds column c's 32 squares in row order starting from 0 --
// the fixed float32 order the score definition uses.  In QDQ mode (the
// trainer's W4A16 fake quantization, [QUADS] 2.2 A) each element's dequantized
// value fl(level * d_b) is also stored, rounded to bf16; codes and scales may
// then be skipped (codes == nullptr).
__device__ __forceinline__ void quantize_block16(const uint4& lo, const uint4& hi, float s_t,
                                                 float* f, BlockScale& bs, uint2& c) {
  bf16x8_to_f32(lo, f);
  bf16x8_to_f32(hi, f + 8);
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(f[j]));
  bs = block_scale(m, s_t);
  c.x = quantize8(f, bs);
  c.y = quantize8(f + 8, bs);
}

// The task loop of one 256-thread block (tasks first, first + stride, ...),
// shared by the quantizer kernel and the fused activation-side kernel; `sq`
// is 32 x 256 floats of shared memory in score mode.
template <bool kScores, bool kQdq>
__device__ __forceinline__ void quantize_block_tasks(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    const int32_t* __restrict__ row_index, const int32_t* __restrict__ goff, int G,
    const float* __restrict__ st, const uint32_t* __restrict__ amax_bits,
    uint8_t* __restrict__ codes, int64_t ldc, uint8_t* __restrict__ scales, int layout,
    float* __restrict__ partials, __nv_bfloat16* __restrict__ qdq, int64_t ldq, float* sq,
    int64_t first, int64_t stride, const float* gscale = nullptr,
    const int32_t* __restrict__ gcnt = nullptr) {
  // tensor scales: a per-block table (gscale, shared memory), given (st), or
  // derived from the groups' amax bits (read through L2: the fused kernel
  // produces them earlier in the same launch)
  auto scale_of = [&](int g) {
    if (gscale) return gscale[g];
    return amax_bits ? tensor_scale_from_amax(__uint_as_float(__ldcg(amax_bits + g))) : __ldcg(st + g);
  };
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t end = goff ? (int64_t)goff[G] : rows;
  if (!QDBG(end >= 0 && end <= rows)) end = 0;
  const int nslab = (cols + 255) >> 8;
  const int64_t nchunks = (end + kScoreChunk - 1) / kScoreChunk;
  const int64_t ntasks = nchunks * nslab;   // < 2^31 (host check)
  const int ncols16 = cols >> 4;
  const int blk = lane & 15;
  // tensor scale of a single group, once per block
  const float s_single = G == 1 ? scale_of(0) : 0.0f;
  // with gcnt, rows of a chunk at or past goff[g] + gcnt[g] (its group's
  // padding) are zero rows: not read (a chunk lies inside one group)
  auto real_end = [&](int64_t r0, int64_t r1) -> int64_t {
    if (!gcnt) return r1;
    const int g = group_of(goff, G, r0);
    return min(r1, (int64_t)goff[g] + gcnt[g]);
  };
  // this thread's two rows of a task, loaded one task ahead (task indices fit
  // in 32 bits: the division is a 32-bit one)
  auto load_task = [&](int64_t task, uint4 (&raw)[2][2]) {
    const uint32_t tk = (uint32_t)task;
    const int64_t chunk = tk / (uint32_t)nslab;
    const int col = (int)(tk - (uint32_t)chunk * (uint32_t)nslab) * 256 + blk * 16;
    const int64_t r0 = chunk * kScoreChunk;
    const int64_t r1 = task < ntasks ? real_end(r0, min(r0 + kScoreChunk, end)) : r0;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int64_t row = r0 + 4 * warp + 2 * it + (lane >> 4);
      raw[it][0] = raw[it][1] = make_uint4(0, 0, 0, 0);
      if (task < ntasks && col < cols && row < r1) {
        const int64_t src = row_index ? (int64_t)row_index[row] : row;
        const uint4* px = reinterpret_cast<const uint4*>(x + src * ldx + col);
        raw[it][0] = __ldg(px);
        raw[it][1] = __ldg(px + 1);
      }
    }
  };
  uint4 nxt[2][2];
  load_task(first, nxt);
  for (int64_t task = first; task < ntasks; task += stride) {
    uint4 raw[2][2];
#pragma unroll
    for (int it = 0; it < 2; ++it) { raw[it][0] = nxt[it][0]; raw[it][1] = nxt[it][1]; }
    load_task(task + stride, nxt);
    const int64_t chunk = (uint32_t)task / (uint32_t)nslab;
    const int slab = (int)((uint32_t)task - (uint32_t)chunk * (uint32_t)nslab);
    const int col = slab * 256 + blk * 16;
    const bool active = col < cols;
    const int64_t r0 = chunk * kScoreChunk;
    const int64_t r1 = min(r0 + kScoreChunk, end);
    const int g0 = goff ? group_of(goff, G, r0) : 0;   // same for the whole block
    if (gcnt && (int64_t)goff[g0] + gcnt[g0] <= r0) {
      // the whole chunk is group padding: the outputs of zero rows (codes,
      // scale bytes, QDQ values and residual partials all 0), nothing read
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int64_t row = r0 + 4 * warp + 2 * it + (lane >> 4);
        if (!active || row >= r1) continue;
        if (!kQdq || codes) {
          uint32_t* pc = reinterpret_cast<uint32_t*>(codes + row * ldc + (col >> 1));
          pc[0] = 0u;
          pc[1] = 0u;
          scales[sf_offset(layout, row, col >> 4, ncols16)] = 0;
        }
        if (kQdq) {
          uint4* pq = reinterpret_cast<uint4*>(qdq + row * ldq + col);
          pq[0] = pq[1] = make_uint4(0, 0, 0, 0);
        }
      }
      if (kScores) {
        const int c = slab * 256 + (int)threadIdx.x;
        if (c < cols) partials[chunk * cols + c] = 0.0f;
      }
      continue;
    }
    const float s_t0 = G == 1 ? s_single : scale_of(g0);
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int64_t row = r0 + 4 * warp + 2 * it + (lane >> 4);
      const bool valid = active && row < r1;
      int g = g0;
      if (goff && valid)
        while (g + 1 < G && row >= goff[g + 1]) ++g;
      float f[16];
      BlockScale bs;
      uint2 c;
      quantize_block16(raw[it][0], raw[it][1], !valid ? 1.0f : g == g0 ? s_t0 : scale_of(g), f, bs,
                       c);
      if (valid && (!kQdq || codes)) {
        uint32_t* pc = reinterpret_cast<uint32_t*>(codes + row * ldc + (col >> 1));
        pc[0] = c.x;
        pc[1] = c.y;
        scales[sf_offset(layout, row, col >> 4, ncols16)] = (uint8_t)bs.byte;
      }
      if (kQdq && valid) {
        float lv[16];
        e2m1x8_to_f32(c.x, lv);
        e2m1x8_to_f32(c.y, lv + 8);
        uint32_t packed[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(lv[2 * j], bs.d),
                                                   __fmul_rn(lv[2 * j + 1], bs.d));
          packed[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        uint4* pq = reinterpret_cast<uint4*>(qdq + row * ldq + col);
        pq[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        pq[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      }
      if (kScores) {
        float lv[16];
        e2m1x8_to_f32(c.x, lv);
        e2m1x8_to_f32(c.y, lv + 8);
        float4* ps = reinterpret_cast<float4*>(sq + (row - r0) * 256 + blk * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // rows past the end were loaded as zeros: their codes and R are 0
            const float R = __fsub_rn(f[4 * q + j], __fmul_rn(lv[4 * q + j], bs.d));
            v[j] = __fmul_rn(R, R);
          }
          // 16-byte chunk q of this block lands at chunk q ^ ((blk >> 1) & 3): the
          // eight lanes of a store phase then cover all 32 banks
          ps[q ^ ((blk >> 1) & 3)] = make_float4(v[0], v[1], v[2], v[3]);
        }
      }
    }
    if (kScores) {
      __syncthreads();
      const int c = slab * 256 + (int)threadIdx.x;
      if (c < cols) {
        float acc = 0.0f;
        const int nr = (int)(r1 - r0);
        // column c sits at its swizzled position (chunk of 4 within its 16-block)
        const int cb = (int)threadIdx.x >> 4;
        const int pc = ((int)threadIdx.x & ~15) | (((((int)threadIdx.x >> 2) & 3) ^ ((cb >> 1) & 3)) << 2) |
                       ((int)threadIdx.x & 3);
        for (int r = 0; r < nr; ++r) acc = __fadd_rn(acc, sq[r * 256 + pc]);
        partials[chunk * cols + c] = acc;
      }
      __syncthreads();
    }
  }
}


// Score mode: four blocks per SM (64 registers, no spills); the others
// three (85 registers, no spills at 64).
template <bool kScores, bool kQdq>
__global__ void __launch_bounds__(256, kScores ? 4 : 3) quantize_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    const int32_t* __restrict__ row_index, const int32_t* __restrict__ goff, int G,
    const float* __restrict__ st, const uint32_t* __restrict__ amax_bits, float* __restrict__ st_out,
    uint8_t* __restrict__ codes, int64_t ldc, uint8_t* __restrict__ scales, int layout,
    float* __restrict__ partials, __nv_bfloat16* __restrict__ qdq, int64_t ldq,
    const int32_t* __restrict__ gcnt) {
  griddep_wait();
  __shared__ __align__(16) float sq[kScores ? kScoreChunk * 256 : 4];
  // groups (up to kSmemGroups): offsets and tensor scales once per block in
  // shared memory, so the per-task group search and scale reads stay on chip
  __shared__ int32_t s_goff[kSmemGroups + 1];
  __shared__ float s_scale[kSmemGroups];
  __shared__ int32_t s_cnt[kSmemGroups];
  // tensor scales derived from the groups' amax bits are also stored by block 0
  if (amax_bits && blockIdx.x == 0)
    for (int g = threadIdx.x; g < G; g += blockDim.x)
      st_out[g] = tensor_scale_from_amax(__uint_as_float(__ldg(amax_bits + g)));
  const bool cache = goff && G <= kSmemGroups;
  if (cache) {
    for (int g = threadIdx.x; g <= G; g += blockDim.x) s_goff[g] = goff[g];
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
      s_scale[g] = amax_bits ? tensor_scale_from_amax(__uint_as_float(__ldg(amax_bits + g))) : __ldg(st + g);
      if (gcnt) s_cnt[g] = __ldg(gcnt + g);
    }
    __syncthreads();
  }
  quantize_block_tasks<kScores, kQdq>(x, rows, cols, ldx, row_index, cache ? s_goff : goff, G, st,
                                      amax_bits, codes, ldc, scales, layout, partials, qdq, ldq, sq,
                                      blockIdx.x, gridDim.x, cache ? s_scale : nullptr,
                                      cache && gcnt ? s_cnt : gcnt);
}

// Score mode with one thread per (32-row chunk, 16-column block): the thread
// walks its chunk's rows in order (the next D rows' loads in flight), writes
// each row's codes and block scale, and adds each column's residual square to
// a register in row order from 0 -- the same float32 sequence the shared-
// memory column sums form -- so the partials need no shared memory and no
// barrier.  Chunks never straddle a group (group offsets are multiples of 32
// in score mode).  Used when there are enough (chunk, block) pairs to fill
// the GPU.  D = 2 at three blocks per SM, D = 4 at two (more bytes in flight
// per SM; chosen when every resident thread gets several pairs, since one
// wave fewer threads otherwise leaves a tail).
template <int D>
__global__ void __launch_bounds__(256, D == 2 ? 3 : 2) quantize_chunk_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    const int32_t* __restrict__ row_index, const int32_t* __restrict__ goff, int G,
    const float* __restrict__ st, const uint32_t* __restrict__ amax_bits, float* __restrict__ st_out,
    uint8_t* __restrict__ codes, int64_t ldc, uint8_t* __restrict__ scales, int layout,
    float* __restrict__ partials, const int32_t* __restrict__ gcnt) {
  griddep_wait();
  __shared__ int32_t s_goff[kSmemGroups + 1];
  __shared__ float s_scale[kSmemGroups];
  __shared__ int32_t s_cnt[kSmemGroups];
  if (amax_bits && blockIdx.x == 0)
    for (int g = threadIdx.x; g < G; g += blockDim.x)
      st_out[g] = tensor_scale_from_amax(__uint_as_float(__ldg(amax_bits + g)));
  const bool cache = G <= kSmemGroups;
  if (cache) {
    if (goff)
      for (int g = threadIdx.x; g <= G; g += blockDim.x) s_goff[g] = goff[g];
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
      s_scale[g] = amax_bits ? tensor_scale_from_amax(__uint_as_float(__ldg(amax_bits + g))) : __ldg(st + g);
      if (gcnt) s_cnt[g] = __ldg(gcnt + g);
    }
    __syncthreads();
  }
  const int32_t* go = cache ? s_goff : goff;
  const int32_t* gc = cache && gcnt ? s_cnt : gcnt;
  auto scale_of = [&](int g) {
    if (cache) return s_scale[g];
    return amax_bits ? tensor_scale_from_amax(__uint_as_float(__ldcg(amax_bits + g))) : __ldg(st + g);
  };
  int64_t end = goff ? (int64_t)go[G] : rows;
  if (!QDBG(end >= 0 && end <= rows)) end = 0;
  const uint32_t nblk = (uint32_t)cols >> 4;
  const uint32_t total = (uint32_t)(((end + kScoreChunk - 1) / kScoreChunk) * nblk);   // < 2^31 (host check)
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const uint32_t chunk = i / nblk, cb = i - chunk * nblk;
    const int64_t r0 = (int64_t)chunk * kScoreChunk;
    const int nr = (int)min((int64_t)kScoreChunk, end - r0);
    const int g = goff ? group_of(go, G, r0) : 0;
    if (goff && r0 + nr > (int64_t)go[g + 1]) atomicExch(&g_quant_error, QUADS_ERR_DEVICE_CHECK);
    // rows of the chunk past its group's count (gcnt) are zero rows: not read
    const int nreal = gc ? (int)max((int64_t)0, min((int64_t)nr, (int64_t)go[g] + gc[g] - r0)) : nr;
    if (nreal == 0 && nr > 0) {
      // the whole chunk is group padding: zero codes, scale bytes and partials
      for (int r = 0; r < nr; ++r) {
        *reinterpret_cast<uint2*>(codes + (r0 + r) * ldc + cb * 8) = make_uint2(0u, 0u);
        scales[sf_offset(layout, r0 + r, cb, nblk)] = 0;
      }
      float4* pz = reinterpret_cast<float4*>(partials + (int64_t)chunk * cols + cb * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) pz[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    const float s_t = scale_of(g);
    auto load = [&](int r, uint4& lo, uint4& hi) {
      if (r < nreal) {
        const int64_t src = row_index ? (int64_t)row_index[r0 + r] : r0 + r;
        const uint4* px = reinterpret_cast<const uint4*>(x + src * ldx + cb * 16);
        lo = __ldg(px);
        hi = __ldg(px + 1);
      } else {
        lo = hi = make_uint4(0, 0, 0, 0);   // padding (or past the chunk): a zero row
      }
    };
    uint4 bl[D], bh[D];   // rows r .. r + D - 1, row r + q in slot (r + q) % D
#pragma unroll
    for (int q = 0; q < D; ++q) load(q, bl[q], bh[q]);
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
#pragma unroll 1
    for (int rb = 0; rb < nr; rb += D) {
#pragma unroll
    for (int q = 0; q < D; ++q) {
      const int r = rb + q;
      if (r >= nr) break;
      const uint4 lo = bl[q], hi = bh[q];
      load(r + D, bl[q], bh[q]);
      const int64_t row = r0 + r;
      float f[16];
      BlockScale bs;
      uint2 c;
      quantize_block16(lo, hi, s_t, f, bs, c);
      *reinterpret_cast<uint2*>(codes + row * ldc + cb * 8) = c;
      scales[sf_offset(layout, row, cb, nblk)] = (uint8_t)bs.byte;
      float lv[16];
      e2m1x8_to_f32(c.x, lv);
      e2m1x8_to_f32(c.y, lv + 8);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float R = __fsub_rn(f[j], __fmul_rn(lv[j], bs.d));
        acc[j] = __fadd_rn(acc[j], __fmul_rn(R, R));
      }
    }
    }
    float4* pp = reinterpret_cast<float4*>(partials + (int64_t)chunk * cols + cb * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) pp[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  }
}

// ---------------------------------------------------------------- select
// Channel scores = the group's chunk partials added in ascending chunk order
// starting from 0 (one float32 add per chunk).  Two launch shapes compute the
// same sequence of adds:
//  * long groups (many chunks): a block owns 32 channels of one group; each
//    slice of up to 256 chunks is staged in shared memory by all warps
//    (coalesced reads, 8 in flight per thread), then lane l of warp 0 adds
//    channel l's chunks in order;
//  * short groups: inside the top-k kernel, one thread per (group, channel)
//    loops over the chunks.
__global__ void __launch_bounds__(256) score_chain_kernel(const float* __restrict__ partials,
                                                          int cols,
                                                          const int32_t* __restrict__ goff,
                                                          int64_t rows,
                                                          float* __restrict__ scores) {
  griddep_wait();
  __shared__ float tile[256][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = blockIdx.y;
  const int c = blockIdx.x * 32 + lane;
  const int64_t a = goff ? (int64_t)goff[g] : 0;
  const int64_t b = goff ? (int64_t)goff[g + 1] : rows;
  const int64_t c0 = a / kScoreChunk, c1 = (b + kScoreChunk - 1) / kScoreChunk;
  float t = 0.0f;  // warp 0: running total of channel c
  for (int64_t base = c0; base < c1; base += 256) {
    const int n = (int)min((int64_t)256, c1 - base);
    // every thread stages rows warp, warp+8, ... of the slice, 8 loads in flight
#pragma unroll
    for (int j0 = 0; j0 < 32; j0 += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = warp + 8 * (j0 + j);
        v[j] = (i < n && c < cols) ? __ldg(partials + (base + i) * cols + c) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) tile[warp + 8 * (j0 + j)][lane] = v[j];
    }
    __syncthreads();
    if (warp == 0)
      for (int i = 0; i < n; ++i) t = __fadd_rn(t, tile[i][lane]);
    __syncthreads();
  }
  if (warp == 0 && c < cols) scores[(int64_t)g * cols + c] = t;
}


// Top-k of `cols` keys held PER per thread by a block of NT threads (key i of
// thread t is channel t*PER + i): radix selection on the bit patterns (scores
// are >= 0, so the unsigned order of the bits is the float order) finds the
// k-th largest key T byte by byte; the channels with key > T and the
// lowest-index channels with key == T are written to sel_out in ascending
// order.  Each of the four byte passes has its own histogram (zeroed up
// front), so a pass costs two block barriers (histogram complete; warp 0 has
// found the byte); the output positions come from one block-wide scan of the
// per-thread (key > T, key == T) counts.  Shared scratch: hist[4*256],
// warp_tot[NT/32], dn[2].
template <int NT, int PER>
__device__ __forceinline__ void block_topk(const uint32_t (&key)[PER], int cols, int k,
                                           int32_t* sel_out, int* hist, int* warp_tot, int* dn) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 4 * 256; i += NT) hist[i] = 0;
  __syncthreads();
  uint32_t prefix = 0u, mask_hi = 0u;   // bytes fixed so far
  int need = k;                         // how many of the keys matching prefix are still taken
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int* h = hist + 256 * pass;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int c = threadIdx.x * PER + i;
      if (c < cols && (key[i] & mask_hi) == prefix) atomicAdd(&h[(key[i] >> shift) & 255u], 1);
    }
    __syncthreads();
    if (w == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending); the bin in which the
      // running count from the top reaches `need` holds the k-th key
      int c8[8], lsum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { c8[i] = h[255 - 8 * lane - i]; lsum += c8[i]; }
      int incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const int excl = incl - lsum;
      const unsigned found = __ballot_sync(0xffffffffu, excl < need && incl >= need);
      if (lane == __ffs(found) - 1) {
        int nd = need - excl, i = 0;
        for (; i < 7; ++i) {
          if (c8[i] >= nd) break;
          nd -= c8[i];
        }
        dn[0] = 255 - 8 * lane - i;
        dn[1] = nd;
      }
    }
    __syncthreads();
    // dn is rewritten only after the next pass's first barrier, which every
    // thread reaches after this read
    prefix |= (uint32_t)dn[0] << shift;
    need = dn[1];
    mask_hi |= 255u << shift;
  }
  // selected: key > T, and the first `need` channels (in index order) with key == T
  const uint32_t T = prefix;
  int ngt = 0, neq = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int c = threadIdx.x * PER + i;
    ngt += (c < cols && key[i] > T) ? 1 : 0;
    neq += (c < cols && key[i] == T) ? 1 : 0;
  }
  // both counts in one word (each total <= cols <= 65535): exclusive block scan
  const int v = (ngt << 16) | neq;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int j = 0; j < NW; ++j)
    if (j < w) before += warp_tot[j];
  const int ex = before + incl - v;
  int gt_b = ex >> 16, eq_b = ex & 0xffff;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int c = threadIdx.x * PER + i;
    if (c < cols && key[i] > T) {
      sel_out[gt_b + min(eq_b, need)] = c;
      ++gt_b;
    } else if (c < cols && key[i] == T) {
      if (eq_b < need) sel_out[gt_b + eq_b] = c;
      ++eq_b;
    }
  }
}

// Top-k per group by radix selection on the score bit patterns (scores are
// >= 0, so the unsigned order of the bits is the float order): find the k-th
// largest key T byte by byte, take every channel with key > T and the
// lowest-index channels with key == T, and write them in ascending order.
// With `partials` (short groups) the block first forms its group's scores
// itself -- the chunk partials added in ascending chunk order from 0 -- and
// stores them to `scores`; otherwise it reads the scores score_chain_kernel
// left there.
// NT threads x PER channels per thread cover cols: 256 x 8 up to 2048
// precomputed scores, 256 x 4 up to 1024 and 1024 x 2 up to 2048 channels
// formed from partials, 1024 x 8 up to 8192 (a barrier costs more with more
// warps; more threads keep more partial loads in flight).
template <int NT, int PER, int U>
__global__ void __launch_bounds__(NT) topk_kernel(float* __restrict__ scores, int cols,
                                                  int k, int32_t* __restrict__ sel,
                                                  const float* __restrict__ partials,
                                                  const int32_t* __restrict__ goff,
                                                  int64_t rows) {
  griddep_wait();
  __shared__ int hist[4 * 256];
  __shared__ int warp_tot[NT / 32];
  __shared__ int dn[2];
  const int g = blockIdx.y;
  float* sc = scores + (int64_t)g * cols;
  uint32_t key[PER];
  if (partials) {
    const int64_t a = goff ? (int64_t)goff[g] : 0;
    const int64_t b = goff ? (int64_t)goff[g + 1] : rows;
    const int64_t c0 = a / kScoreChunk, c1 = (b + kScoreChunk - 1) / kScoreChunk;
    // every column of the thread advances together, U chunks at a time, so
    // that PER x U loads are in flight per round (the round trips, not the
    // adds, set this phase's time); each column's sum still adds its chunks
    // in ascending order
    float t[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) t[i] = 0.0f;
    for (int64_t ch = c0; ch < c1; ch += U) {
      float v[PER][U];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int c = threadIdx.x * PER + i;
#pragma unroll
        for (int u = 0; u < U; ++u)
          v[i][u] = (c < cols && ch + u < c1) ? __ldg(partials + (ch + u) * cols + c) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < PER; ++i)
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (ch + u < c1) t[i] = __fadd_rn(t[i], v[i][u]);
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int c = threadIdx.x * PER + i;
      if (c < cols) sc[c] = t[i];
      key[i] = c < cols ? __float_as_uint(t[i]) : 0u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int c = threadIdx.x * PER + i;
      key[i] = c < cols ? __float_as_uint(sc[c]) : 0u;
    }
  }
  block_topk<NT, PER>(key, cols, k, sel + (int64_t)g * k, hist, warp_tot, dn);
}

// ---------------------------------------------------------------- residual slice
// Block-scale table of one tensor scale s_t: for every E4M3 byte, d =
// E4M3 * s_t and its correctly rounded reciprocal (0 where the block's codes
// are 0), so that a gathered element needs two shared loads instead of the
// per-element scale decode.
__device__ __forceinline__ void fill_scale_table(float s_t, float* td, float* tr) {
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    const BlockScale bs = block_scale_from_byte((uint32_t)b, s_t);
    td[b] = bs.d;
    tr[b] = bs.zero ? 0.0f : bs.r;   // d is finite, so 1/d == 0 only for zero blocks
  }
}
// R = x - fl(DQ(Q(x))) for two elements with their blocks' table entries:
// the code is the E2M1 rounding of fl(x * r) (0 where r == 0), as
// quantize_block16 forms it.
__device__ __forceinline__ void residual_pair(float xa, float xb, uint32_t sa, uint32_t sb,
                                              const float* td, const float* tr, float& Ra,
                                              float& Rb) {
  const float ra = tr[sa], rb = tr[sb];
  float qa, qb;
  e2m1_round_pair(__fmul_rn(xa, ra), __fmul_rn(xb, rb), qa, qb);
  if (ra == 0.0f) qa = 0.0f;
  if (rb == 0.0f) qb = 0.0f;
  Ra = __fsub_rn(xa, __fmul_rn(qa, td[sa]));
  Rb = __fsub_rn(xb, __fmul_rn(qb, td[sb]));
}

// R[:, sel] recomputed from x and the stored block scales; one block per
// slice of `rb` rows (8 or 32: group offsets are multiples of 32, so a slice
// is inside one group; 8 when 32-row slices would leave the GPU short of
// blocks), four independent gathers in flight per thread; per-group amax of
// |R| by atomicMax on the float bits.
__global__ void __launch_bounds__(256) rsel_residual_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    const int32_t* __restrict__ goff, int G, const int32_t* __restrict__ gcnt,
    const uint8_t* __restrict__ scales, int layout,
    const float* __restrict__ st, const int32_t* __restrict__ sel, int k,
    float* __restrict__ rs, uint32_t* __restrict__ amax_bits, int rb) {
  griddep_wait();
  __shared__ float red[8];
  __shared__ float td[256], tr[256];
  const int64_t end = goff ? (int64_t)goff[G] : rows;
  const int64_t nblk = (end + rb - 1) / rb;
  const int ncols16 = cols >> 4;
  int tab_g = -1;
  for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int64_t r0 = blk * rb, r1 = min(r0 + rb, end);
    const int g = goff ? group_of(goff, G, r0) : 0;
    if (g != tab_g) {   // block-uniform: the scale table of the slice's group
      __syncthreads();
      fill_scale_table(st[g], td, tr);
      __syncthreads();
      tab_g = g;
    }
    const int32_t* sg = sel + (int64_t)g * k;
    // rows of the slice past its group's count (gcnt) are zero rows: not read
    const int64_t rr = gcnt ? max(r0, min(r1, (int64_t)goff[g] + gcnt[g])) : r1;
    float m = 0.0f;
    const int total = (int)(r1 - r0) * k;
    for (int i0 = threadIdx.x; i0 < total; i0 += 4 * blockDim.x) {
      int64_t r[4];
      int j[4], c[4];
      float xv[4];
      uint32_t sb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        r[u] = r0 + (i < total ? i / k : 0);
        j[u] = i < total ? i % k : 0;
        c[u] = sg[j[u]];
        if (!QDBG(c[u] >= 0 && c[u] < cols)) c[u] = 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool real = r[u] < rr;   // a zero row: x = 0 and scale byte 0, so R = 0
        xv[u] = real ? __bfloat162float(x[r[u] * ldx + c[u]]) : 0.0f;
        sb[u] = real ? scales[sf_offset(layout, r[u], c[u] >> 4, ncols16)] : 0u;
      }
      float R[4];
      residual_pair(xv[0], xv[1], sb[0], sb[1], td, tr, R[0], R[1]);
      residual_pair(xv[2], xv[3], sb[2], sb[3], td, tr, R[2], R[3]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        if (i >= total) continue;
        rs[r[u] * k + j[u]] = R[u];
        m = fmaxf(m, fabsf(R[u]));
      }
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
      float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
      v = warp_max(v);
      if (threadIdx.x == 0 && v > 0.0f) atomicMax(&amax_bits[g], __float_as_uint(v));
    }
    __syncthreads();
  }
}

// Per-group path (many groups, e.g. one per expert): one block per group does
// both steps -- R for the group's rows into the float32 workspace, the
// group's amax by a block reduction, then the second quantization of those
// rows (the arithmetic of rsel_residual_kernel and rsel_quantize_kernel) --
// so no grid-wide maximum and no second launch are needed.  Blocks past the
// groups zero the rows after the last offset.
constexpr int kRselGroupThreads = 1024;

// Zero R_sel codes and scales of rows [end, rows) (past the last group), as
// block `b` of `nb` blocks.
__device__ __forceinline__ void rsel_zero_tail(int64_t rows, int64_t end, int kpad,
                                               uint8_t* __restrict__ rcodes,
                                               uint8_t* __restrict__ rscales, int rlayout, int b,
                                               int nb) {
  const int vpr = kpad >> 3, rcols16 = kpad >> 4;
  const int64_t total = (rows - end) * vpr;
  for (int64_t i = (int64_t)b * blockDim.x + threadIdx.x; i < total; i += (int64_t)nb * blockDim.x) {
    const int64_t r = end + i / vpr;
    const int col = (int)(i % vpr) * 8;
    *reinterpret_cast<uint32_t*>(rcodes + r * (kpad >> 1) + (col >> 1)) = 0u;
    if (((col >> 3) & 1) == 0) rscales[sf_offset(rlayout, r, col >> 4, rcols16)] = 0;
  }
}

// R[:, sel] of one group's rows [r0, r1) by the whole block: R into the
// float32 workspace rs (row r at rs + r * k), the group's amax by a block
// reduction, then the second quantization of those rows.  Rows at or past
// rreal are zero rows (not read; their R is 0).  td/tr: the block-scale table
// of the group's tensor scale (filled, and a barrier passed, by the caller);
// sg: the group's k selected channels; red: NT/32 floats of shared memory.
// The group's R_sel tensor scale is stored to *rst_g.  Optional on-chip
// copies (shared memory, row r at r - r0) replace the global reads and the
// workspace: xs the rows' bf16 values (row stride cols), ss their scale
// bytes (row stride cols/16), rsm R itself (row stride k).
__device__ __forceinline__ void rsel_group_rows(
    const __nv_bfloat16* __restrict__ x, int cols, int64_t ldx, int64_t r0, int64_t r1,
    int64_t rreal, const uint8_t* scales, int layout, const int32_t* sg, int k, int kpad,
    float* rs, uint8_t* __restrict__ rcodes, uint8_t* __restrict__ rscales, int rlayout,
    float* rst_g, const float* td, const float* tr, float* red,
    const __nv_bfloat16* xs = nullptr, const uint8_t* ss = nullptr, float* rsm = nullptr) {
  const int ncols16 = cols >> 4, rcols16 = kpad >> 4;
  const int vpr = kpad >> 3;   // 8-element vectors per residual row (even)
  // rows past rreal: R = 0, so only the real rows are gathered (four
  // independent gathers in flight per thread)
  const int total = (int)(rreal - r0) * k;
  float m = 0.0f;
  for (int i0 = threadIdx.x; i0 < total; i0 += 4 * blockDim.x) {
    int rl[4], j[4], c[4];
    float xv[4];
    uint32_t sb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      rl[u] = i < total ? i / k : 0;
      j[u] = i < total ? i - rl[u] * k : 0;
      c[u] = sg[j[u]];
      if (!QDBG(c[u] >= 0 && c[u] < cols)) c[u] = 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (xs) {
        xv[u] = __bfloat162float(xs[(int64_t)rl[u] * cols + c[u]]);
        sb[u] = ss[(int64_t)rl[u] * ncols16 + (c[u] >> 4)];
      } else {
        const int64_t r = r0 + rl[u];
        xv[u] = __bfloat162float(x[r * ldx + c[u]]);
        sb[u] = scales[sf_offset(layout, r, c[u] >> 4, ncols16)];
      }
    }
    float R[4];
    residual_pair(xv[0], xv[1], sb[0], sb[1], td, tr, R[0], R[1]);
    residual_pair(xv[2], xv[3], sb[2], sb[3], td, tr, R[2], R[3]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      if (i >= total) continue;
      if (rsm) rsm[(int64_t)rl[u] * k + j[u]] = R[u];
      else rs[(r0 + rl[u]) * k + j[u]] = R[u];
      m = fmaxf(m, fabsf(R[u]));
    }
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();   // also makes this block's rs writes visible to the block
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float rs_t = tensor_scale_from_amax(red[0]);
  if (threadIdx.x == 0) *rst_g = rs_t;
  const int nvec = (int)(r1 - r0) * vpr;   // < 2^31: rows * k is (host check)
  // warp-uniform loop: lanes 2i / 2i+1 hold the two halves of one 16-block
  for (int base = (int)(threadIdx.x & ~31u); base < nvec; base += blockDim.x) {
    const int i = base + (int)(threadIdx.x & 31);
    const bool in = i < nvec;
    const int rq = in ? i / vpr : 0;
    const int64_t r = r0 + rq;
    const int col = in ? (i - rq * vpr) * 8 : 0;
    const bool live = in && col < k && r < rreal;   // rows past rreal: R = 0
    float f[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) f[jj] = 0.0f;
    if (live) {
      const float4* p = reinterpret_cast<const float4*>(rsm ? rsm + (r - r0) * k + col : rs + r * k + col);
      const float4 a = p[0], b = p[1];
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
      f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    float mm = 0.0f;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) mm = fmaxf(mm, fabsf(f[jj]));
    mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 1));
    const BlockScale bs = block_scale(mm, rs_t);
    uint32_t cw = quantize8(f, bs);
    uint32_t sbyte = bs.byte;
    if (!live) { cw = 0u; sbyte = 0u; }
    if (in) {
      *reinterpret_cast<uint32_t*>(rcodes + r * (kpad >> 1) + (col >> 1)) = cw;
      if (((col >> 3) & 1) == 0) rscales[sf_offset(rlayout, r, col >> 4, rcols16)] = (uint8_t)sbyte;
    }
  }
}

__global__ void __launch_bounds__(kRselGroupThreads) rsel_group_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    const int32_t* __restrict__ goff, int G, const int32_t* __restrict__ gcnt,
    const uint8_t* __restrict__ scales, int layout,
    const float* __restrict__ st, const int32_t* __restrict__ sel, int k, int kpad,
    float* __restrict__ rs, uint8_t* __restrict__ rcodes, uint8_t* __restrict__ rscales,
    int rlayout, float* __restrict__ rst) {
  griddep_wait();
  __shared__ float red[kRselGroupThreads / 32];
  if ((int)blockIdx.x >= G) {
    // rows past the last offset: zero codes and scales
    rsel_zero_tail(rows, goff[G], kpad, rcodes, rscales, rlayout, (int)blockIdx.x - G,
                   (int)gridDim.x - G);
    return;
  }
  const int g = blockIdx.x;
  const int64_t r0 = goff[g], r1 = goff[g + 1];
  __shared__ float td[256], tr[256];
  fill_scale_table(st[g], td, tr);
  __syncthreads();
  // rows past the group's count (gcnt) are zero rows: not read
  const int64_t rr = gcnt ? r0 + min(max((int64_t)gcnt[g], (int64_t)0), r1 - r0) : r1;
  rsel_group_rows(x, cols, ldx, r0, r1, rr, scales, layout, sel + (int64_t)g * k, k, kpad, rs,
                  rcodes, rscales, rlayout, rst + g, td, tr, red);
}

// ---------------------------------------------------------------- per-group quantize + select
// One block per group (the MoE layer's h: one per expert) does the whole
// activation side of that group -- RTN quantization of its rows with the
// residual energies, the channel scores, the top-k selection, the residual
// slice R[:, sel] and its second quantization.  Groups are independent, so
// nothing waits on another block, the chunk partials never leave the block,
// and R_sel's gather finds the group's rows in L2 right after they were read.
// Phase 1 takes the group's 32-row chunks in order: thread t quantizes the
// chunk's (row, 16-column block) items t and t + NT (the next chunk's rows
// are loaded meanwhile) and parks each residual square in shared memory;
// after a barrier thread c adds column c's 32 squares in row order from 0 and
// adds that chunk partial to its running score -- the float32 sequence of the
// score definition (chunk partials in ascending chunk order from 0).  Chunks
// past the group's count are padding: zero codes and scales, and a partial
// of 0, which leaves the score as it is.  Phase 2 is the block top-k of the
// other select paths, phase 3 the per-group R_sel of rsel_group_kernel.  A
// group of at most stash_rows real rows (decode-sized) also keeps its rows
// and their scale bytes in shared memory during phase 1, and R in the
// squares' buffer during phase 3, so R_sel reads nothing from memory.
constexpr int kQsgThreads = 1024;
constexpr int kQsgMaxCols = 1024;   // one channel per thread; 32 x cols floats of shared memory
__global__ void __launch_bounds__(kQsgThreads, 1) quantize_select_groups_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    const int32_t* __restrict__ goff, int G, const int32_t* __restrict__ gcnt,
    const float* __restrict__ st_in, const float* __restrict__ amax_in, uint8_t* codes,
    int64_t ldc, uint8_t* scales, int layout, float* __restrict__ st_out, int k, int kpad,
    int32_t* __restrict__ sel, float* __restrict__ scores_out, float* rs,
    uint8_t* __restrict__ rcodes, uint8_t* __restrict__ rscales, int rlayout,
    float* __restrict__ rst, int stash_rows) {
  griddep_wait();
  // residual squares of one chunk, [32][cols]: the four 4-column quarters of a
  // 16-block at quarter q ^ ((block >> 1) & 3), so that the eight lanes of a
  // 16-byte store phase and the 32 lanes of a column read hit distinct banks;
  // then [stash_rows][cols] bf16 rows and [stash_rows][cols/16] scale bytes
  extern __shared__ __align__(16) float sq[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(sq + kScoreChunk * cols);
  uint8_t* ss = reinterpret_cast<uint8_t*>(xs + (int64_t)stash_rows * cols);
  __shared__ int hist[4 * 256];
  __shared__ int warp_tot[kQsgThreads / 32];
  __shared__ int dn[2];
  __shared__ int32_t s_sel[kQsgMaxCols];
  __shared__ float td[256], tr[256], red[kQsgThreads / 32];
  if ((int)blockIdx.x >= G) {
    // rows past the last offset: zero R_sel codes and scales
    rsel_zero_tail(rows, goff[G], kpad, rcodes, rscales, rlayout, (int)blockIdx.x - G,
                   (int)gridDim.x - G);
    return;
  }
  const int g = blockIdx.x;
  const int64_t r0 = goff[g], r1 = goff[g + 1];
  if (!QDBG(r0 >= 0 && r1 >= r0 && r1 <= rows)) return;
  // chunks are the score definition's 32-row chunks only when groups start
  // at multiples of 32
  if (threadIdx.x == 0 && r0 % kScoreChunk) atomicExch(&g_quant_error, QUADS_ERR_DEVICE_CHECK);
  // rows at or past rr are zero rows: not read
  const int64_t rr = gcnt ? r0 + min(max((int64_t)gcnt[g], (int64_t)0), r1 - r0) : r1;
  const int ncols16 = cols >> 4;
  const bool stash = rr - r0 <= stash_rows;

  // ---- tensor scale: given, from the given amax, or from the group's own amax
  float s_t;
  if (st_in) {
    s_t = st_in[g];
  } else if (amax_in) {
    s_t = tensor_scale_from_amax(amax_in[g]);
  } else {
    const int vpr = cols >> 3;
    const int64_t nv = (rr - r0) * vpr;
    __nv_bfloat162 m2 = __floats2bfloat162_rn(0.0f, 0.0f);
    for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) {
      const int64_t rl = i / vpr;
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + (r0 + rl) * ldx) + (i - rl * vpr));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[j])));
    }
    const float2 mf = __bfloat1622float2(m2);
    const float m = warp_max(fmaxf(mf.x, mf.y));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float v = 0.0f;
#pragma unroll 1
    for (int j = 0; j < (int)(blockDim.x >> 5); ++j) v = fmaxf(v, red[j]);
    s_t = tensor_scale_from_amax(v);
    __syncthreads();   // red is reused below
  }
  if (threadIdx.x == 0) st_out[g] = s_t;

  // ---- phase 1: quantization and channel scores
  const int items = kScoreChunk * ncols16;   // (row, block) items per chunk, <= 2 * kQsgThreads
  const int64_t nreal = (rr - r0 + kScoreChunk - 1) / kScoreChunk;   // chunks holding real rows
  // this thread's two items of every chunk: row in the chunk and 16-block
  int irl[2], icb[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int it = (int)threadIdx.x + u * kQsgThreads;
    irl[u] = it < items ? it / ncols16 : kScoreChunk;   // kScoreChunk: no item
    icb[u] = it < items ? it - irl[u] * ncols16 : 0;
  }
  auto load_chunk = [&](int64_t ch, uint4 (&raw)[2][2]) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      raw[u][0] = raw[u][1] = make_uint4(0, 0, 0, 0);
      const int64_t row = r0 + ch * kScoreChunk + irl[u];
      if (ch < nreal && irl[u] < kScoreChunk && row < rr) {
        const uint4* px = reinterpret_cast<const uint4*>(x + row * ldx + icb[u] * 16);
        raw[u][0] = __ldg(px);
        raw[u][1] = __ldg(px + 1);
      }
    }
  };
  float score = 0.0f;   // channel threadIdx.x
  uint4 nxt[2][2];
  load_chunk(0, nxt);
#pragma unroll 1
  for (int64_t ch = 0; ch < nreal; ++ch) {
    uint4 raw[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) { raw[u][0] = nxt[u][0]; raw[u][1] = nxt[u][1]; }
    load_chunk(ch + 1, nxt);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (irl[u] >= kScoreChunk) continue;
      const int rl = irl[u], cb = icb[u];
      const int64_t row = r0 + ch * kScoreChunk + rl;
      float f[16];
      BlockScale bs;
      uint2 c;
      // rows past rr were loaded as zeros: codes, scale byte and R are 0
      quantize_block16(raw[u][0], raw[u][1], s_t, f, bs, c);
      if (row < r1) {
        uint32_t* pc = reinterpret_cast<uint32_t*>(codes + row * ldc + cb * 8);
        pc[0] = c.x;
        pc[1] = c.y;
        scales[sf_offset(layout, row, cb, ncols16)] = (uint8_t)bs.byte;
      }
      if (stash && row < rr) {
        uint4* px = reinterpret_cast<uint4*>(xs + (row - r0) * cols + cb * 16);
        px[0] = raw[u][0];
        px[1] = raw[u][1];
        ss[(row - r0) * ncols16 + cb] = (uint8_t)bs.byte;
      }
      float lv[16];
      e2m1x8_to_f32(c.x, lv);
      e2m1x8_to_f32(c.y, lv + 8);
      float4* ps = reinterpret_cast<float4*>(sq + rl * cols + cb * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float R = __fsub_rn(f[4 * q + j], __fmul_rn(lv[4 * q + j], bs.d));
          v[j] = __fmul_rn(R, R);
        }
        ps[q ^ ((cb >> 1) & 3)] = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
    __syncthreads();
    if ((int)threadIdx.x < cols) {
      const int c = threadIdx.x, cb = c >> 4;
      const int pc = (c & ~15) | ((((c >> 2) & 3) ^ ((cb >> 1) & 3)) << 2) | (c & 3);
      float acc = 0.0f;
#pragma unroll 8
      for (int r = 0; r < kScoreChunk; ++r) acc = __fadd_rn(acc, sq[r * cols + pc]);
      score = __fadd_rn(score, acc);
    }
    __syncthreads();
  }
  // padding chunks: the outputs of zero rows (a warp per row, lanes over its 16-blocks)
  {
    const int64_t p0 = r0 + nreal * kScoreChunk;
    const int nw = (int)(blockDim.x >> 5), lane = (int)(threadIdx.x & 31);
    for (int64_t row = p0 + (threadIdx.x >> 5); row < r1; row += nw) {
      for (int cb = lane; cb < ncols16; cb += 32) {
        uint32_t* pc = reinterpret_cast<uint32_t*>(codes + row * ldc + cb * 8);
        pc[0] = 0u;
        pc[1] = 0u;
        scales[sf_offset(layout, row, cb, ncols16)] = 0;
      }
    }
  }
  if (scores_out && (int)threadIdx.x < cols) scores_out[(int64_t)g * cols + threadIdx.x] = score;

  // ---- phase 2: top-k channels of the group (ascending)
  {
    const uint32_t key[1] = {(int)threadIdx.x < cols ? __float_as_uint(score) : 0u};
    block_topk<kQsgThreads, 1>(key, cols, k, s_sel, hist, warp_tot, dn);
  }
  // ---- phase 3: R[:, sel] and its second quantization
  fill_scale_table(s_t, td, tr);
  __syncthreads();   // s_sel, the table, and this block's code and scale stores are visible
  for (int j = threadIdx.x; j < k; j += blockDim.x) sel[(int64_t)g * k + j] = s_sel[j];
  // R fits the squares' buffer when (real rows) * k <= 32 * cols
  float* rsm = (rr - r0) * k <= (int64_t)kScoreChunk * cols ? sq : nullptr;
  rsel_group_rows(x, cols, ldx, r0, r1, rr, scales, layout, s_sel, k, kpad, rs, rcodes, rscales,
                  rlayout, rst + g, td, tr, red, stash ? xs : nullptr, stash ? ss : nullptr, rsm);
}

// Quantize the float32 residual slice [rows, k] (16-blocks along the selection)
// into codes [rows, kpad/2] and scales (kpad columns, padding blocks 0).
// One thread per 8 elements; lanes 2i/2i+1 share a block.
__global__ void __launch_bounds__(256) rsel_quantize_kernel(
    const float* __restrict__ rs, int64_t rows, int k, int kpad, const int32_t* __restrict__ goff,
    int G, const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ rcodes,
    uint8_t* __restrict__ rscales, int layout, float* __restrict__ rst) {
  griddep_wait();
  const int64_t end = goff ? (int64_t)goff[G] : rows;
  const int vec_per_row = kpad >> 3;  // even
  const int64_t total = rows * vec_per_row;  // padding rows (>= end) get zeros
  const int ncols16 = kpad >> 4;
  if (blockIdx.x == 0)
    for (int g = threadIdx.x; g < G; g += blockDim.x)
      rst[g] = tensor_scale_from_amax(__uint_as_float(amax_bits[g]));
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
       i < ((total + 31) / 32) * 32; i += (int64_t)gridDim.x * blockDim.x) {
    const bool in = i < total;
    const int64_t r = in ? i / vec_per_row : 0;
    const int col = in ? (int)(i % vec_per_row) * 8 : 0;
    float f[8];
    const bool live = in && r < end && col < k;
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = 0.0f;
    float s_t = 1.0f;
    if (live) {
      const float4* p = reinterpret_cast<const float4*>(rs + r * k + col);
      const float4 a = p[0], b = p[1];
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
      f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      const int g = goff ? group_of(goff, G, r) : 0;
      s_t = tensor_scale_from_amax(__uint_as_float(amax_bits[g]));
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const BlockScale bs = block_scale(m, s_t);
    uint32_t c = quantize8(f, bs);
    uint32_t sb = bs.byte;
    if (!live) { c = 0u; sb = 0u; }
    if (in) {
      *reinterpret_cast<uint32_t*>(rcodes + r * (kpad >> 1) + (col >> 1)) = c;
      if (((col >> 3) & 1) == 0) rscales[sf_offset(layout, r, col >> 4, ncols16)] = (uint8_t)sb;
    }
  }
}

// ---------------------------------------------------------------- fused activation side
// The whole activation side of one compensated GEMM in one cooperative
// kernel: tensor amax, RTN quantization with the residual-energy partials,
// channel scores, top-k selection, the residual slice R[:, sel] and its second
// quantization -- five phases separated by four grid-wide barriers.  X is read
// from HBM once: the second (quantizing) pass and the gather of the selected
// columns find it in L2 when it fits there (a 8192 x 2048 bf16 activation is
// 32 MiB of the 129 MB L2).  Every block computes the same top-k from the
// same scores, so the selection needs no further barrier.  The barrier waits
// are bounded; a barrier that does not complete latches
// QUADS_ERR_DEVICE_TIMEOUT and the kernel returns.
struct FusedCtl {
  uint32_t amax_x;    // float bits of max |x|
  uint32_t amax_r;    // float bits of max |R_sel|
  uint32_t count;     // barrier arrivals
  uint32_t gen;       // barrier generation
};
constexpr int kFusedThreads = 256;

__device__ __forceinline__ bool grid_barrier(FusedCtl* ctl, unsigned long long tmo, int* err) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint32_t g = *reinterpret_cast<volatile uint32_t*>(&ctl->gen);
    __threadfence();
    if (atomicAdd(&ctl->count, 1u) == gridDim.x - 1) {
      atomicExch(&ctl->count, 0u);
      __threadfence();
      atomicAdd(&ctl->gen, 1u);
    } else {
      unsigned long long t0 = 0;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
      while (*reinterpret_cast<volatile uint32_t*>(&ctl->gen) == g) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > tmo) {
          ok = 0;
          atomicExch(err, QUADS_ERR_DEVICE_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

template <int PER>
__global__ void __launch_bounds__(kFusedThreads, 4) quantize_select_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    uint8_t* __restrict__ codes, int64_t ldc, uint8_t* __restrict__ scales, int layout,
    float* __restrict__ st_out, float* __restrict__ partials,
    float* __restrict__ scores, int k, int kpad, int32_t* __restrict__ sel, float* __restrict__ rs,
    uint8_t* __restrict__ rcodes, uint8_t* __restrict__ rscales, int rlayout,
    float* __restrict__ rst, FusedCtl* ctl, unsigned long long tmo) {
  // phase B's residual squares (32 x 256) and phase C's partial tile (256 x 33)
  // share one buffer
  __shared__ __align__(16) float sbuf[256 * 33];
  float (*tile)[33] = reinterpret_cast<float (*)[33]>(sbuf);
  __shared__ int hist[4 * 256];
  __shared__ int warp_tot[kFusedThreads / 32];
  __shared__ int dn[2];
  __shared__ int32_t s_sel[kFusedMaxK];
  __shared__ float red[kFusedThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kFusedThreads / 32;
  const int ncols16 = cols >> 4;

  // ---- A: tensor amax (exact maximum of bf16 magnitudes)
  {
    const int vpr = cols >> 3;
    const int64_t nvec = rows * vpr;
    __nv_bfloat162 m2 = __floats2bfloat162_rn(0.0f, 0.0f);
    const int64_t stride = (int64_t)gridDim.x * kFusedThreads;
    for (int64_t i0 = (int64_t)blockIdx.x * kFusedThreads + threadIdx.x; i0 < nvec; i0 += 4 * stride) {
      uint4 u[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t i = i0 + q * stride;
        u[q] = make_uint4(0, 0, 0, 0);
        if (i < nvec) {
          const int64_t r = i / vpr;
          u[q] = __ldg(reinterpret_cast<const uint4*>(x + r * ldx) + (i - r * vpr));
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[j])));
      }
    }
    const float2 mf = __bfloat1622float2(m2);
    float m = warp_max(fmaxf(mf.x, mf.y));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
      float v = lane < NW ? red[lane] : 0.0f;
      v = warp_max(v);
      if (lane == 0 && v > 0.0f) atomicMax(&ctl->amax_x, __float_as_uint(v));
    }
  }
  if (!grid_barrier(ctl, tmo, &g_quant_error)) return;

  // ---- B: quantization and residual-energy partials
  if (blockIdx.x == 0 && threadIdx.x == 0)
    st_out[0] = tensor_scale_from_amax(__uint_as_float(*reinterpret_cast<volatile uint32_t*>(&ctl->amax_x)));
  quantize_block_tasks<true, false>(x, rows, cols, ldx, nullptr, nullptr, 1, nullptr, &ctl->amax_x,
                                    codes, ldc, scales, layout, partials, nullptr, 0, sbuf,
                                    blockIdx.x, gridDim.x);
  if (!grid_barrier(ctl, tmo, &g_quant_error)) return;

  // ---- C: channel scores = chunk partials added in ascending chunk order
  {
    const int64_t nchunks = (rows + kScoreChunk - 1) / kScoreChunk;
    for (int cg = blockIdx.x; cg * 32 < cols; cg += gridDim.x) {
      const int c = cg * 32 + lane;
      float t = 0.0f;
      for (int64_t base = 0; base < nchunks; base += 256) {
        const int n = (int)min((int64_t)256, nchunks - base);
#pragma unroll
        for (int j = 0; j < 256 / NW; ++j) {
          const int i = warp + NW * j;
          tile[i][lane] = (i < n && c < cols) ? __ldcg(partials + (base + i) * cols + c) : 0.0f;
        }
        __syncthreads();
        if (warp == 0)
          for (int i = 0; i < n; ++i) t = __fadd_rn(t, tile[i][lane]);
        __syncthreads();
      }
      if (warp == 0 && c < cols) scores[c] = t;
    }
  }
  if (!grid_barrier(ctl, tmo, &g_quant_error)) return;

  // ---- D: every block selects the same top-k; R[:, sel] of this block's rows
  {
    uint32_t key[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int c = threadIdx.x * PER + i;
      key[i] = c < cols ? __float_as_uint(__ldcg(scores + c)) : 0u;
    }
    block_topk<kFusedThreads, PER>(key, cols, k, s_sel, hist, warp_tot, dn);
    __syncthreads();
    if (blockIdx.x == 0)
      for (int j = threadIdx.x; j < k; j += kFusedThreads) sel[j] = s_sel[j];
    const float s_t = tensor_scale_from_amax(__uint_as_float(*reinterpret_cast<volatile uint32_t*>(&ctl->amax_x)));
    const int64_t rpb = (rows + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = min(rows, (int64_t)blockIdx.x * rpb), r1 = min(rows, r0 + rpb);
    const int64_t total = (r1 - r0) * k;
    float m = 0.0f;
    for (int64_t i = threadIdx.x; i < total; i += kFusedThreads) {
      const int64_t r = r0 + i / k;
      const int j = (int)(i % k);
      int c = s_sel[j];
      if (!QDBG(c >= 0 && c < cols)) c = 0;
      const float xv = __bfloat162float(x[r * ldx + c]);
      const BlockScale bs =
          block_scale_from_byte(__ldcg(scales + sf_offset(layout, r, c >> 4, ncols16)), s_t);
      float v[8] = {__fmul_rn(xv, bs.r), 0, 0, 0, 0, 0, 0, 0};
      const uint32_t code = bs.zero ? 0u : (f32x8_to_e2m1(v) & 15u);
      const float R = __fsub_rn(xv, __fmul_rn(e2m1_to_f32(code), bs.d));
      rs[r * k + j] = R;
      m = fmaxf(m, fabsf(R));
    }
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
      float v = lane < NW ? red[lane] : 0.0f;
      v = warp_max(v);
      if (lane == 0 && v > 0.0f) atomicMax(&ctl->amax_r, __float_as_uint(v));
    }
  }
  if (!grid_barrier(ctl, tmo, &g_quant_error)) return;

  // ---- E: second quantization of this block's rows of R_sel (own tensor scale)
  {
    const float rs_t = tensor_scale_from_amax(__uint_as_float(*reinterpret_cast<volatile uint32_t*>(&ctl->amax_r)));
    if (blockIdx.x == 0 && threadIdx.x == 0) rst[0] = rs_t;
    const int rcols16 = kpad >> 4;
    const int vpr = kpad >> 3;   // 8-element vectors per residual row (even)
    const int64_t rpb = (rows + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = min(rows, (int64_t)blockIdx.x * rpb), r1 = min(rows, r0 + rpb);
    const int64_t nvec = (r1 - r0) * vpr;
    // warp-uniform loop: lanes 2i / 2i+1 hold the two halves of one 16-block
    for (int64_t base = (int64_t)warp * 32; base < nvec; base += kFusedThreads) {
      const int64_t i = base + lane;
      const bool in = i < nvec;
      const int64_t r = r0 + (in ? i / vpr : 0);
      const int col = in ? (int)(i % vpr) * 8 : 0;
      const bool live = in && col < k;
      float f[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) f[jj] = 0.0f;
      if (live) {
        const float4* pp = reinterpret_cast<const float4*>(rs + r * k + col);
        const float4 a = __ldcg(pp), b = __ldcg(pp + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      }
      float mm = 0.0f;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) mm = fmaxf(mm, fabsf(f[jj]));
      mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, 1));
      const BlockScale bs = block_scale(mm, rs_t);
      uint32_t cw = quantize8(f, bs);
      uint32_t sbyte = bs.byte;
      if (!live) { cw = 0u; sbyte = 0u; }
      if (in) {
        *reinterpret_cast<uint32_t*>(rcodes + r * (kpad >> 1) + (col >> 1)) = cw;
        if (((col >> 3) & 1) == 0) rscales[sf_offset(rlayout, r, col >> 4, rcols16)] = (uint8_t)sbyte;
      }
    }
  }
}

// ---------------------------------------------------------------- TRACE
// Word-parallel form of the rule.  With n = the RTN code of v (same sign as v;
// a zero result keeps the sign of v) and its magnitude level m_n, the two
// neighbours of v are n itself and, when v is not a level, the code one
// magnitude step away from zero (|v| > |q_n|) or toward zero (|v| < |q_n|),
// with the same sign (a step toward zero from magnitude 1 gives a zero that
// keeps the sign of v).  Nearest to the rollout code r (values compared, +0 ==
// -0) is the neighbour step when
//   away from zero:  r has the sign of n and a larger magnitude;
//   toward zero:     r has the other sign, or a smaller magnitude,
// else n.  (|v| > 6 rounds to 6 and no magnitude is larger; |v| < |q_n| needs
// m_n >= 1.)  Eight 4-bit codes are handled at once in a 32-bit word with
// per-nibble arithmetic that never carries across nibbles.

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// Sign bits of eight floats to bit 4j: the top bytes of the even and of the
// odd elements are gathered into one word each (byte permutes), whose sign
// bits then sit at 8k + 7 for elements 2k and 2k + 1.
__device__ __forceinline__ uint32_t sign_nibbles8(const float* d) {
  const uint32_t e = prmt(prmt(__float_as_uint(d[0]), __float_as_uint(d[2]), 0x0073u),
                          prmt(__float_as_uint(d[4]), __float_as_uint(d[6]), 0x0073u), 0x5410u);
  const uint32_t o = prmt(prmt(__float_as_uint(d[1]), __float_as_uint(d[3]), 0x0073u),
                          prmt(__float_as_uint(d[5]), __float_as_uint(d[7]), 0x0073u), 0x5410u);
  return ((e >> 7) & 0x01010101u) | ((o >> 3) & 0x10101010u);
}

// Per element, whether |v| lies beyond its RTN level (away) or inside it
// (toward): bit 4j of the returned masks.  |v| - |q| is exact whenever the
// two are within a factor of two (Sterbenz) and otherwise far from zero, so
// its sign decides; equal magnitudes give +0 in both differences.
__device__ __forceinline__ void trace_dirs8(const float* v, const float* qn, uint32_t& away,
                                            uint32_t& toward) {
  float a[8], b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a[j] = __fsub_rn(fabsf(v[j]), fabsf(qn[j]));   // < 0: toward zero
    b[j] = __fsub_rn(fabsf(qn[j]), fabsf(v[j]));   // < 0: away from zero
  }
  toward = sign_nibbles8(a);
  away = sign_nibbles8(b);
}

constexpr uint32_t kNib1 = 0x11111111u, kNib7 = 0x77777777u, kNib8 = 0x88888888u;

// Nibbles of x that are zero, as bit 4j.
__device__ __forceinline__ uint32_t zero_nibbles(uint32_t x) {
  x |= x >> 2;
  x |= x >> 1;
  return ~x & kNib1;
}

// TRACE codes of eight elements (rtn: RTN codes, rc: rollout codes, dirs from
// trace_dirs8), and the counter contributions: values of RTN != rollout,
// TRACE != rollout, and RTN mismatches one signed level from the rollout.
__device__ __forceinline__ uint32_t trace_word(uint32_t rtn, uint32_t rc, uint32_t away,
                                               uint32_t toward, unsigned& n_rtn, unsigned& n_tr,
                                               unsigned& n_adj) {
  const uint32_t mn = rtn & kNib7, mr = rc & kNib7;
  const uint32_t same = ~((rtn ^ rc) >> 3) & kNib1;          // equal sign bits
  const uint32_t ge_r = (((mr | kNib8) - mn) >> 3) & kNib1;  // m_r >= m_n
  const uint32_t ge_n = (((mn | kNib8) - mr) >> 3) & kNib1;  // m_n >= m_r
  const uint32_t up = away & same & ~ge_n;                   // same sign, m_r > m_n
  const uint32_t dn = toward & (~same | ~ge_r) & kNib1;      // other sign, or m_r < m_n
  const uint32_t out = rtn + up - dn;
  // value mismatch: magnitudes differ, or signs differ on a nonzero magnitude
  const uint32_t nz_n = ((mn + kNib7) >> 3) & kNib1;
  const uint32_t neq = (~zero_nibbles(mn ^ mr) & kNib1) | (~same & nz_n & kNib1);
  // one signed level apart: same sign and |m_n - m_r| == 1, or other signs and
  // m_n + m_r == 1
  const uint32_t e = ((mr | kNib8) - mn) ^ kNib8;            // m_r - m_n mod 16
  const uint32_t neg = (e >> 3) & kNib1;
  const uint32_t absd = (e ^ (neg * 15u)) + neg;             // |m_r - m_n| <= 7
  const uint32_t adj = (same & zero_nibbles(absd ^ kNib1)) | (~same & zero_nibbles((mn + mr) ^ kNib1));
  n_rtn += __popc(neq);
  n_adj += __popc(adj & kNib1);
  n_tr += __popc(neq) - __popc((up | dn) & adj);   // a step onto an adjacent rollout level matches it
  return out;
}

// One thread per 16-element block of a row per step (kMx: per 16 elements of
// a 32-element block), with the next step's loads (x, rollout codes, scale)
// issued before the current block is computed, so that loads stay in flight
// across the arithmetic.
// kMx: MXFP4 rollout (E8M0 scale per 32 elements, no tensor scale): the
// scaled value is x * 2^-e and no block is a zero block.
struct TraceItem {
  uint4 x0, x1;     // 16 bf16
  uint2 rc;         // 16 rollout codes
  uint32_t sbyte;   // block scale byte
};

// Row r and 16-block b of a flat block index, advanced by the grid stride
// (dr rows and db blocks, bpr blocks per row) without a division per step.
__device__ __forceinline__ void row_block_step(uint32_t& r, uint32_t& b, uint32_t dr, uint32_t db,
                                               uint32_t bpr) {
  r += dr;
  b += db;
  if (b >= bpr) {
    b -= bpr;
    ++r;
  }
}

template <bool kMx>
__device__ __forceinline__ void trace_load(TraceItem& it, uint32_t i, uint32_t total, uint32_t r,
                                           uint32_t b, const __nv_bfloat16* xt, int64_t ldx,
                                           const uint8_t* rcodes, int64_t ldc,
                                           const uint8_t* rscales, int cols) {
  if (i >= total) return;
  const int col = (int)b * 16;
  const uint4* px = reinterpret_cast<const uint4*>(xt + (int64_t)r * ldx + col);
  it.x0 = __ldg(px);
  it.x1 = __ldg(px + 1);
  const uint32_t* pc = reinterpret_cast<const uint32_t*>(rcodes + (int64_t)r * ldc + (col >> 1));
  it.rc = make_uint2(__ldg(pc), __ldg(pc + 1));   // 4-byte aligned (ldc % 4 == 0)
  it.sbyte = kMx ? __ldg(rscales + (int64_t)r * (cols >> 5) + (col >> 5))
                 : __ldg(rscales + (int64_t)r * (cols >> 4) + (col >> 4));
}

// Five blocks per SM (48 registers, no spills).
template <bool kMx>
__global__ void __launch_bounds__(256, 5) trace_kernel(
    const __nv_bfloat16* __restrict__ xt, int64_t rows, int cols, int64_t ldx,
    const uint8_t* __restrict__ rcodes, int64_t ldc, const uint8_t* __restrict__ rscales,
    const float* __restrict__ rst, uint8_t* __restrict__ out,
    unsigned long long* __restrict__ counters) {
  const uint32_t blk_per_row = (uint32_t)cols >> 4;
  const uint32_t total = (uint32_t)(rows * blk_per_row);   // < 2^31 (host check)
  const uint32_t stride = gridDim.x * blockDim.x;
  // NVFP4: 1/d of every scale byte under the tensor scale (0 for a zero
  // block), so a block needs one shared load instead of the scale decode and
  // the correctly rounded reciprocal
  __shared__ float td[kMx ? 1 : 256], tr[kMx ? 1 : 256];
  if (!kMx) {
    fill_scale_table(rst[0], td, tr);
    __syncthreads();
  }
  unsigned int n_rtn = 0, n_tr = 0, n_adj = 0;
  uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t dr = stride / blk_per_row, db = stride - dr * blk_per_row;
  uint32_t nr = i / blk_per_row, nb = i - nr * blk_per_row;   // the next load's row and block
  TraceItem nxt;
  trace_load<kMx>(nxt, i, total, nr, nb, xt, ldx, rcodes, ldc, rscales, cols);
  for (; i < total; i += stride) {
    const TraceItem cur = nxt;
    const uint32_t r = nr;
    const int col = (int)nb * 16;
    row_block_step(nr, nb, dr, db, blk_per_row);
    trace_load<kMx>(nxt, i + stride, total, nr, nb, xt, ldx, rcodes, ldc, rscales, cols);
    BlockScale bs;
    if (kMx) {
      bs.r = e8m0_inverse(cur.sbyte);
      bs.zero = false;
    } else {
      bs.r = tr[cur.sbyte];
      bs.zero = bs.r == 0.0f;
    }
    uint32_t outw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float f[8];
      bf16x8_to_f32(h ? cur.x1 : cur.x0, f);
      float v[8];
      const uint64_t rr = f2_pack(bs.r, bs.r);
#pragma unroll
      for (int j = 0; j < 8; j += 2) f2_unpack(f2_mul(f2_pack(f[j], f[j + 1]), rr), v[j], v[j + 1]);
      uint32_t rtn = f32x8_to_e2m1(v);
      float qn[8];
      e2m1x8_to_f32(rtn, qn);
      uint32_t away, toward;
      trace_dirs8(v, qn, away, toward);
      if (bs.zero) rtn = away = toward = 0u;   // a zero block gives 0x0 codes
      outw[h] = trace_word(rtn, h ? cur.rc.y : cur.rc.x, away, toward, n_rtn, n_tr, n_adj);
    }
    uint32_t* po = reinterpret_cast<uint32_t*>(out + (int64_t)r * ldc + (col >> 1));
    po[0] = outw[0];
    po[1] = outw[1];
  }
  if (counters) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_rtn += __shfl_xor_sync(0xffffffffu, n_rtn, o);
      n_tr += __shfl_xor_sync(0xffffffffu, n_tr, o);
      n_adj += __shfl_xor_sync(0xffffffffu, n_adj, o);
    }
    if ((threadIdx.x & 31) == 0) {
      if (n_rtn) atomicAdd(&counters[0], (unsigned long long)n_rtn);
      if (n_tr) atomicAdd(&counters[1], (unsigned long long)n_tr);
      if (n_adj) atomicAdd(&counters[2], (unsigned long long)n_adj);
    }
  }
}

// ---------------------------------------------------------------- MXFP4
// MXFP4 quantization (32-element blocks, E8M0 power-of-two scales, no tensor
// scale).  A thread takes 16 elements, half a block; the block maximum comes
// from one shuffle with the partner lane (the even lane writes the scale
// byte).  Scaling by 2^-e is exact, so the codes are the E2M1 rounding
// (ties to even, saturating) of x * 2^-e.  Optional bf16 QDQ output
// level * 2^e (exact in float32).  The loop runs on warp-uniform bases so
// both partners of a block are always active together.
__global__ void __launch_bounds__(256) mx_quantize_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t rows, int cols, int64_t ldx,
    uint8_t* __restrict__ codes, int64_t ldc, uint8_t* __restrict__ scales, int layout,
    __nv_bfloat16* __restrict__ qdq, int64_t ldq) {
  const uint32_t per_row = (uint32_t)cols >> 4;              // even: cols % 32 == 0
  const uint32_t total = (uint32_t)(rows * per_row);         // < 2^31 (host check)
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < total; base += stride) {
    const uint32_t i = base + lane;
    const bool valid = i < total;
    float f[16];
    uint32_t r = 0, h = 0;
    if (valid) {
      r = i / per_row;
      h = i - r * per_row;
      const uint4* px = reinterpret_cast<const uint4*>(x + (int64_t)r * ldx + h * 16);
      bf16x8_to_f32(__ldg(px), f);
      bf16x8_to_f32(__ldg(px + 1), f + 8);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) f[j] = 0.0f;
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(f[j]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    if (!valid) continue;
    const uint32_t byte = e8m0_scale_byte(m);
    const float inv = e8m0_inverse(byte);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(f[j], inv);
    const uint32_t c0 = f32x8_to_e2m1(v), c1 = f32x8_to_e2m1(v + 8);
    *reinterpret_cast<uint2*>(codes + (int64_t)r * ldc + h * 8) = make_uint2(c0, c1);
    if ((h & 1) == 0) scales[sf_offset(layout, r, h >> 1, cols >> 5)] = (uint8_t)byte;
    if (qdq) {
      const float d = e8m0_value(byte);
      float lv[16];
      e2m1x8_to_f32(c0, lv);
      e2m1x8_to_f32(c1, lv + 8);
      uint32_t packed[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(lv[2 * j], d), __fmul_rn(lv[2 * j + 1], d));
        packed[j] = *reinterpret_cast<uint32_t*>(&b2);
      }
      uint4* pq = reinterpret_cast<uint4*>(qdq + (int64_t)r * ldq + h * 16);
      pq[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      pq[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
  }
}

// ---------------------------------------------------------------- TRACE records
// Compact rollout record ([TRACE] "核心方法", "方法步骤详情" step 2): of each
// rollout code only its mantissa bit (the low bit of the 3 magnitude bits) is
// kept, 8 per byte, element 8i+j in bit j of byte i; with the E4M3 block scale
// (8 bits per 16 values) that is the pages' 1.5 bits per value.
// One thread per 8 codes: a 4-byte read, a 1-byte write.
// Bit 0 of each of the eight nibbles of c, as bits 0..7.
__device__ __forceinline__ uint32_t gather_nibble_bit0(uint32_t c) {
  c &= 0x11111111u;
  c = (c | (c >> 3)) & 0x03030303u;
  c = (c | (c >> 6)) & 0x000F000Fu;
  return (c | (c >> 12)) & 0xFFu;
}

// One thread per 32 codes (a 16-byte read, a 4-byte write) when the row
// length allows it (vec), else per 8 codes (a 4-byte read, a 1-byte write).
__global__ void __launch_bounds__(256) trace_pack_kernel(const uint8_t* __restrict__ codes,
                                                         int64_t rows, int cols, int64_t ldc,
                                                         uint8_t* __restrict__ bits,
                                                         int64_t ldb, int vec) {
  const uint32_t per_row = (uint32_t)cols >> (vec ? 5 : 3);
  const uint32_t total = (uint32_t)(rows * per_row);   // < 2^31 (host check)
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const uint32_t r = i / per_row, v = i - r * per_row;
    if (vec) {
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(codes + (int64_t)r * ldc) + v);
      const uint32_t m = gather_nibble_bit0(c.x) | (gather_nibble_bit0(c.y) << 8) |
                         (gather_nibble_bit0(c.z) << 16) | (gather_nibble_bit0(c.w) << 24);
      *reinterpret_cast<uint32_t*>(bits + (int64_t)r * ldb + 4 * v) = m;
    } else {
      const uint32_t c = __ldg(reinterpret_cast<const uint32_t*>(codes + (int64_t)r * ldc) + v);
      bits[(int64_t)r * ldb + v] = (uint8_t)gather_nibble_bit0(c);
    }
  }
}

// Rounding guided by the 1-bit record: of the two E2M1 neighbours of v =
// x_train / d_b (rollout scale), adjacent levels have opposite mantissa bits,
// so the record bit names one of them -- the rollout's own code whenever it
// is one of the two (the off-by-one case the pages find in over 99% of
// mismatches).  A v on a level (or clamped at +-6) has that level alone.
// Counters (nullable, added to): #(result != RTN code), #(result's mantissa
// bit != record bit).
// Eight record bits (element j in bit j) spread to bit 4j.
__device__ __forceinline__ uint32_t spread_bits8(uint32_t b) {
  b = (b | (b << 12)) & 0x000F000Fu;
  b = (b | (b << 6)) & 0x03030303u;
  b = (b | (b << 3)) & 0x11111111u;
  return b;
}

// TRACE from the 1-bit record: the two neighbours of v (when v is not a
// level) are adjacent signed levels with opposite mantissa bits, so the one
// named by the record bit is the RTN code n when n's mantissa bit matches,
// else the neighbour step (away from or toward zero, as in trace_word).
__global__ void __launch_bounds__(256) trace_1bit_kernel(
    const __nv_bfloat16* __restrict__ xt, int64_t rows, int cols, int64_t ldx,
    const uint8_t* __restrict__ mbits, int64_t ldb, const uint8_t* __restrict__ rscales,
    const float* __restrict__ rst, uint8_t* __restrict__ out, int64_t ldc,
    unsigned long long* __restrict__ counters) {
  // one 16-element block per thread and step, the next step's loads issued
  // before the current block is computed (as in trace_kernel)
  const uint32_t blk_per_row = (uint32_t)cols >> 4;
  const uint32_t total = (uint32_t)(rows * blk_per_row);   // < 2^31 (host check)
  const uint32_t stride = gridDim.x * blockDim.x;
  // 1/d of every scale byte (0 for a zero block), as in trace_kernel
  __shared__ float td[256], tr[256];
  fill_scale_table(rst[0], td, tr);
  __syncthreads();
  unsigned int n_chg = 0, n_bit = 0;
  auto load = [&](uint32_t i, uint32_t r, uint32_t bi, uint4& x0, uint4& x1, uint32_t& mb,
                  uint32_t& sb) {
    if (i >= total) return;
    const uint4* px = reinterpret_cast<const uint4*>(xt + (int64_t)r * ldx + bi * 16);
    x0 = __ldg(px);
    x1 = __ldg(px + 1);
    const uint8_t* pb = mbits + (int64_t)r * ldb + bi * 2;
    mb = (uint32_t)__ldg(pb) | ((uint32_t)__ldg(pb + 1) << 8);
    sb = __ldg(rscales + (int64_t)r * (cols >> 4) + bi);
  };
  uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t dr = stride / blk_per_row, db = stride - dr * blk_per_row;
  uint32_t nr = i / blk_per_row, nb = i - nr * blk_per_row;   // the next load's row and block
  uint4 nx0 = make_uint4(0, 0, 0, 0), nx1 = nx0;
  uint32_t nmb = 0, nsb = 0;
  load(i, nr, nb, nx0, nx1, nmb, nsb);
  for (; i < total; i += stride) {
    const uint4 x0 = nx0, x1 = nx1;
    const uint32_t mb16 = nmb, sbyte = nsb;
    const uint32_t r = nr, bi = nb;
    row_block_step(nr, nb, dr, db, blk_per_row);
    load(i + stride, nr, nb, nx0, nx1, nmb, nsb);
    BlockScale bs;
    bs.r = tr[sbyte];
    bs.zero = bs.r == 0.0f;
    uint32_t outw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float f[8];
      bf16x8_to_f32(h ? x1 : x0, f);
      float v[8];
      const uint64_t rr = f2_pack(bs.r, bs.r);
#pragma unroll
      for (int j = 0; j < 8; j += 2) f2_unpack(f2_mul(f2_pack(f[j], f[j + 1]), rr), v[j], v[j + 1]);
      uint32_t rtn = f32x8_to_e2m1(v);
      float qn[8];
      e2m1x8_to_f32(rtn, qn);
      uint32_t away, toward;
      trace_dirs8(v, qn, away, toward);
      if (bs.zero) rtn = away = toward = 0u;   // a zero block gives 0x0 codes
      const uint32_t bits = spread_bits8((mb16 >> (8 * h)) & 0xFFu);
      const uint32_t flip = (rtn ^ bits) & kNib1;   // RTN's mantissa bit is not the record's
      // |v| beyond 6 rounds to magnitude 7 and has no level further out
      const uint32_t top = rtn & (rtn >> 1) & (rtn >> 2) & kNib1;
      const uint32_t up = away & flip & ~top, dn = toward & flip;
      const uint32_t w = rtn + up - dn;
      n_chg += __popc(up | dn);
      n_bit += __popc((w ^ bits) & kNib1);
      outw[h] = w;
    }
    uint32_t* po = reinterpret_cast<uint32_t*>(out + (int64_t)r * ldc + bi * 8);
    po[0] = outw[0];
    po[1] = outw[1];
  }
  if (counters) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_chg += __shfl_xor_sync(0xffffffffu, n_chg, o);
      n_bit += __shfl_xor_sync(0xffffffffu, n_bit, o);
    }
    if ((threadIdx.x & 31) == 0) {
      if (n_chg) atomicAdd(&counters[0], (unsigned long long)n_chg);
      if (n_bit) atomicAdd(&counters[1], (unsigned long long)n_bit);
    }
  }
}

// ---------------------------------------------------------------- host side
static int grid_for(int64_t work_items, int per_block, int max_blocks_per_sm = 8) {
  int64_t b = (work_items + per_block - 1) / per_block;
  int64_t cap = (int64_t)num_sms() * max_blocks_per_sm;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return (int)b;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int read_quant_device_error(cudaStream_t) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, g_quant_error, sizeof(int));
  int zero = 0;
  cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(int));
  return v;
}

}  // namespace quads

using namespace quads;

// Shared by the quantizer and the W4A16 QDQ entry points (qdq == nullptr:
// codes and scales only; codes == nullptr: bf16 QDQ values only).
static quads_status_t quantize_impl(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* row_index,
    const int32_t* group_offsets, int32_t num_groups, const int32_t* group_counts,
    const float* tensor_scale_in,
    const float* tensor_amax_in, uint8_t* codes, int64_t ld_codes, uint8_t* scales,
    int32_t scale_layout, float* tensor_scale_out, float* score_partials,
    __nv_bfloat16* qdq, int64_t ldq, void* workspace, size_t workspace_bytes, void* stream) {
  if (rows > 0 && (!x || (!codes && !qdq) || (codes && !scales) || !tensor_scale_out))
    return fail(QUADS_ERR_INVALID_ARG, "quantize: null x/codes/scales/tensor_scale_out");
  if (qdq && (ldq < cols || ldq % 8 || !aligned16(qdq)))
    return fail(QUADS_ERR_MISALIGNED, "qdq: y must be 16-byte aligned with ldy >= cols, ldy %% 8 == 0");
  if (!codes) ld_codes = cols / 2;
  if (rows < 0 || cols <= 0 || cols % 16)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize: cols=%lld must be a positive multiple of 16", (long long)cols);
  if (scale_layout == QUADS_SCALES_TCGEN05 && cols % 64)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize: TCGEN05 scale layout needs cols %% 64 == 0");
  if (scale_layout != QUADS_SCALES_LINEAR && scale_layout != QUADS_SCALES_TCGEN05)
    return fail(QUADS_ERR_INVALID_ARG, "quantize: bad scale_layout %d", scale_layout);
  if (ldx < cols || ldx % 8 || ld_codes < cols / 2 || ld_codes % 4)
    return fail(QUADS_ERR_MISALIGNED, "quantize: ldx=%lld (>=cols, %%8) ld_codes=%lld (>=cols/2, %%4)", (long long)ldx, (long long)ld_codes);
  if (!aligned16(x) || (codes && !aligned16(codes)) ||
      (score_partials && !aligned16(score_partials)))
    return fail(QUADS_ERR_MISALIGNED, "quantize: x/codes/score_partials must be 16-byte aligned");
  const int G = group_offsets ? num_groups : 1;
  if (group_offsets && num_groups < 1) return fail(QUADS_ERR_INVALID_ARG, "quantize: num_groups < 1");
  if (group_counts && !group_offsets)
    return fail(QUADS_ERR_INVALID_ARG, "quantize: group_counts needs group_offsets");
  if (tensor_scale_in && tensor_amax_in)
    return fail(QUADS_ERR_INVALID_ARG, "quantize: give tensor_scale_in or tensor_amax_in, not both");
  if (rows == 0) return QUADS_OK;
  if (!tensor_scale_in && !tensor_amax_in && (workspace_bytes < (size_t)G * 4 || !workspace))
    return fail(QUADS_ERR_WORKSPACE, "quantize: workspace needs %d bytes", G * 4);
  if (!aligned16(workspace)) return fail(QUADS_ERR_MISALIGNED, "quantize: workspace must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const float* stp = tensor_scale_in;
  const uint32_t* amax_bits = nullptr;   // set: the quantize kernel derives the tensor scales
  int launched = 1;
  if (tensor_amax_in) {
    amax_bits = (const uint32_t*)tensor_amax_in;
  } else if (!tensor_scale_in) {
    launched = 2;
    uint32_t* amax = (uint32_t*)workspace;
    cudaMemsetAsync(amax, 0, (size_t)G * 4, st);
    launch_dep(amax_kernel, grid_for((rows + kAmaxRows - 1) / kAmaxRows, 1, 8), 256, 0, st,
        (const __nv_bfloat16*)x, rows, (int)cols, ldx, row_index, group_offsets, G, amax,
        group_counts);
    amax_bits = amax;
  } else if (tensor_scale_in != tensor_scale_out) {
    cudaMemcpyAsync(tensor_scale_out, tensor_scale_in, (size_t)G * 4, cudaMemcpyDeviceToDevice, st);
  }
  if (codes && scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
    // padding rows of the last 128-row block must read as scale 0
    const int64_t ncols16 = cols / 16;
    const int64_t start = (rows / 128) * (ncols16 / 4) * 512;
    cudaMemsetAsync(scales + start, 0, (size_t)(sf_tc_bytes(rows, cols) - start), st);
  }
  const int64_t ntasks = ((rows + 31) / 32) * ((cols + 255) / 256);
  if (ntasks >= (1ll << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize: more than 2^31 32x256 tasks");
  // one resident wave of blocks looping over the tasks (the next task's rows
  // are loaded while the current one is quantized; a block's setup is paid
  // once): 1 GiB plain 282 -> 270 us, 8192 x 2048 plain 20.3 -> 17.9 us
  // against a block per task
  const int per_sm = score_partials ? 4 : 3;
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(ntasks, (int64_t)num_sms() * per_sm));
  const __nv_bfloat16* xb = (const __nv_bfloat16*)x;
  if (qdq)
    launch_dep(quantize_kernel<false, true>, blocks, 256, 0, st,
        xb, rows, (int)cols, ldx, row_index, group_offsets, G, stp, amax_bits, tensor_scale_out,
        codes, ld_codes, scales, scale_layout, nullptr, qdq, ldq, group_counts);
  else if (score_partials && ((rows + 31) / 32) * (cols / 16) >= (int64_t)num_sms() * 512 &&
           ((rows + 31) / 32) * (cols / 16) < (1ll << 31) && ld_codes % 8 == 0) {
    // enough (chunk, block) pairs for a thread each: about two blocks per SM
    // (its 8-byte code stores need ld_codes % 8 == 0; the 32x256-task kernel
    // stores 4 bytes at a time).  Four rows in flight when every resident
    // thread gets at least three pairs (65536 x 2048: 91 -> 80 us; the 8192-
    // token layer's h, about 1.3 pairs a thread, keeps two: 52 vs 58 us)
    const int64_t pairs = ((rows + 31) / 32) * (cols / 16);
    if (pairs >= (int64_t)num_sms() * 2 * 256 * 3)
      launch_dep(quantize_chunk_kernel<4>, grid_for(pairs, 256, 2), 256, 0, st,
          xb, rows, (int)cols, ldx, row_index, group_offsets, G, stp, amax_bits, tensor_scale_out,
          codes, ld_codes, scales, scale_layout, score_partials, group_counts);
    else
      launch_dep(quantize_chunk_kernel<2>, grid_for(pairs, 256, 3), 256, 0, st,
          xb, rows, (int)cols, ldx, row_index, group_offsets, G, stp, amax_bits, tensor_scale_out,
          codes, ld_codes, scales, scale_layout, score_partials, group_counts);
  }
  else if (score_partials)
    launch_dep(quantize_kernel<true, false>, blocks, 256, 0, st,
        xb, rows, (int)cols, ldx, row_index, group_offsets, G, stp, amax_bits, tensor_scale_out,
        codes, ld_codes, scales, scale_layout, score_partials, nullptr, 0, group_counts);
  else
    launch_dep(quantize_kernel<false, false>, blocks, 256, 0, st,
        xb, rows, (int)cols, ldx, row_index, group_offsets, G, stp, amax_bits, tensor_scale_out,
        codes, ld_codes, scales, scale_layout, nullptr, nullptr, 0, group_counts);
  return check_launch(qdq ? "qdq" : "quantize", launched);
}

extern "C" quads_status_t quads_quantize_nvfp4(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* row_index,
    const int32_t* group_offsets, int32_t num_groups, const int32_t* group_counts,
    const float* tensor_scale_in, const float* tensor_amax_in, uint8_t* codes, int64_t ld_codes,
    uint8_t* scales, int32_t scale_layout, float* tensor_scale_out, float* score_partials,
    void* workspace, size_t workspace_bytes, void* stream) {
  if (!codes && rows > 0) return fail(QUADS_ERR_INVALID_ARG, "quantize: null codes");
  return quantize_impl(x, rows, cols, ldx, row_index, group_offsets, num_groups, group_counts,
                       tensor_scale_in, tensor_amax_in, codes, ld_codes, scales, scale_layout,
                       tensor_scale_out, score_partials, nullptr, 0, workspace, workspace_bytes,
                       stream);
}

extern "C" quads_status_t quads_qdq_nvfp4(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* group_offsets,
    int32_t num_groups, const float* tensor_scale_in, void* y, int64_t ldy, uint8_t* codes,
    int64_t ld_codes, uint8_t* scales, int32_t scale_layout, float* tensor_scale_out,
    void* workspace, size_t workspace_bytes, void* stream) {
  if (!y && rows > 0) return fail(QUADS_ERR_INVALID_ARG, "qdq: null y");
  return quantize_impl(x, rows, cols, ldx, nullptr, group_offsets, num_groups, nullptr,
                       tensor_scale_in, nullptr, codes, ld_codes, scales, scale_layout,
                       tensor_scale_out, nullptr, (__nv_bfloat16*)y, ldy, workspace,
                       workspace_bytes, stream);
}

namespace quads {
// Argument checks of the selection call (shared by the workspace and the
// allocation-free entry points, so that both report the same status for the
// same arguments); on success *need is the scratch the call uses.
quads_status_t select_check_args(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                 const int32_t* group_offsets, int32_t num_groups,
                                 const int32_t* group_counts,
                                 const uint8_t* scales, const float* tensor_scale,
                                 const float* score_partials, int32_t k, const int32_t* sel,
                                 const uint8_t* r_codes, const uint8_t* r_scales,
                                 const float* r_tensor_scale, size_t* need) {
  if (rows > 0 && (!x || !scales || !tensor_scale || !score_partials || !sel || !r_codes ||
                   !r_scales || !r_tensor_scale))
    return fail(QUADS_ERR_INVALID_ARG, "select: null pointer argument");
  if (rows < 0 || cols <= 0 || cols % 16 || cols > 8192)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "select: cols=%lld must be a multiple of 16 and <= 8192 (rows >= 0)", (long long)cols);
  if (k <= 0 || k % 16 || k > cols)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "select: k=%d must be a multiple of 16 in [16, cols]", k);
  if (ldx < cols) return fail(QUADS_ERR_MISALIGNED, "select: ldx < cols");
  if ((uintptr_t)r_codes & 15u) return fail(QUADS_ERR_MISALIGNED, "select: r_codes must be 16-byte aligned");
  if (group_offsets && num_groups < 1) return fail(QUADS_ERR_INVALID_ARG, "select: num_groups < 1");
  if (group_counts && !group_offsets)
    return fail(QUADS_ERR_INVALID_ARG, "select: group_counts needs group_offsets");
  *need = quads_workspace_size(QUADS_OP_SELECT, rows, cols, 0, k, group_offsets ? num_groups : 1);
  return QUADS_OK;
}
int debug_line_quantize(long long* value) { return take_debug_line(value); }

}  // namespace quads

extern "C" quads_status_t quads_select_residual_channels(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* group_offsets,
    int32_t num_groups, const int32_t* group_counts, const uint8_t* scales, int32_t scale_layout,
    const float* tensor_scale, const float* score_partials, int32_t k, int32_t* sel,
    float* scores_out, uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout,
    float* r_tensor_scale, void* workspace, size_t workspace_bytes, void* sel_ready_event,
    void* stream) {
  size_t need = 0;
  if (quads_status_t s = select_check_args(x, rows, cols, ldx, group_offsets, num_groups,
                                           group_counts, scales, tensor_scale, score_partials, k,
                                           sel, r_codes, r_scales, r_tensor_scale, &need))
    return s;
  const int G = group_offsets ? num_groups : 1;
  const int kpad = quads_kpad(k);
  if (rows > 0 && (!workspace || workspace_bytes < need))
    return fail(QUADS_ERR_WORKSPACE, "select: workspace needs %zu bytes", need);
  if ((uintptr_t)workspace & 15u) return fail(QUADS_ERR_MISALIGNED, "select: workspace must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  auto sel_ready = [&]() -> quads_status_t {
    if (!sel_ready_event) return QUADS_OK;
    const cudaError_t e = cudaEventRecord((cudaEvent_t)sel_ready_event, st);
    return e == cudaSuccess ? QUADS_OK
                            : fail(QUADS_ERR_CUDA, "select: cudaEventRecord: %s", cudaGetErrorString(e));
  };
  if (rows == 0) return sel_ready();
  float* rs = (float*)workspace;
  const size_t rs_bytes = ((size_t)rows * k * 4 + 255) & ~(size_t)255;
  uint32_t* amax = (uint32_t*)((char*)workspace + rs_bytes);
  float* scores = scores_out ? scores_out
                             : (float*)((char*)workspace + rs_bytes + (((size_t)G * 4 + 255) & ~(size_t)255));
  // chunks per group on average decides the launch shape (both give the same
  // sums); for short groups the top-k block also forms the scores
  const int64_t chunks_per_group = (rows + 31) / 32 / G;
  const bool long_groups = chunks_per_group > 64;
  if (long_groups)
    launch_dep(score_chain_kernel, dim3((unsigned)((cols + 31) / 32), (unsigned)G), 256, 0, st,
        score_partials, (int)cols, group_offsets, rows, scores);
  const float* part = long_groups ? nullptr : score_partials;
  const dim3 tg(1, (unsigned)G);
  if (cols <= 2048 && long_groups)   // scores precomputed: only the selection
    launch_dep(topk_kernel<256, 8, 1>, tg, 256, 0, st,
        scores, (int)cols, k, sel, part, group_offsets, rows);
  else if (cols <= 1024)             // e.g. per-expert h: up to 64 partial loads in flight per thread
    launch_dep(topk_kernel<256, 4, 16>, tg, 256, 0, st,
        scores, (int)cols, k, sel, part, group_offsets, rows);
  else if (cols <= 2048)             // 32 partial loads in flight per thread
    launch_dep(topk_kernel<1024, 2, 16>, tg, 1024, 0, st,
        scores, (int)cols, k, sel, part, group_offsets, rows);
  else
    launch_dep(topk_kernel<1024, 8, 2>, tg, 1024, 0, st,
        scores, (int)cols, k, sel, part, group_offsets, rows);
  if (quads_status_t s = sel_ready()) return s;
  if (group_offsets && G >= kRselGroupMin) {
    if (r_scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
      const int64_t start = (rows / 128) * (kpad / 64) * 512;
      cudaMemsetAsync(r_scales + start, 0, (size_t)(sf_tc_bytes(rows, kpad) - start), st);
    }
    launch_dep(rsel_group_kernel, G + 2 * num_sms(), kRselGroupThreads, 0, st,
        (const __nv_bfloat16*)x, rows, (int)cols, ldx, group_offsets, G, group_counts, scales,
        scale_layout, tensor_scale, sel, k, kpad, rs, r_codes, r_scales, r_scale_layout,
        r_tensor_scale);
    return check_launch("select", long_groups ? 3 : 2);
  }
  cudaMemsetAsync(amax, 0, (size_t)G * 4, st);
  const int rb = (rows + 31) / 32 < 2 * (int64_t)num_sms() ? 8 : 32;
  launch_dep(rsel_residual_kernel, grid_for((rows + rb - 1) / rb, 1, 16), 256, 0, st,
      (const __nv_bfloat16*)x, rows, (int)cols, ldx, group_offsets, G, group_counts, scales,
      scale_layout, tensor_scale, sel, k, rs, amax, rb);
  if (r_scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
    const int64_t start = (rows / 128) * (kpad / 64) * 512;
    cudaMemsetAsync(r_scales + start, 0, (size_t)(sf_tc_bytes(rows, kpad) - start), st);
  }
  launch_dep(rsel_quantize_kernel, grid_for(rows * (kpad / 8), 256), 256, 0, st,
      rs, rows, k, kpad, group_offsets, G, amax, r_codes, r_scales, r_scale_layout, r_tensor_scale);
  return check_launch("select", long_groups ? 4 : 3);
}

extern "C" quads_status_t quads_quantize_select_nvfp4(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, int32_t k, uint8_t* codes,
    int64_t ld_codes, uint8_t* scales, int32_t scale_layout, float* tensor_scale_out, int32_t* sel,
    float* scores_out, uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout,
    float* r_tensor_scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (rows > 0 && (!x || !codes || !scales || !tensor_scale_out || !sel || !r_codes || !r_scales ||
                   !r_tensor_scale))
    return fail(QUADS_ERR_INVALID_ARG, "quantize_select: null pointer argument");
  if (rows < 0 || cols <= 0 || cols % 16 || cols > 8192)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize_select: cols=%lld must be a multiple of 16 and <= 8192", (long long)cols);
  if (k <= 0 || k % 16 || k > cols || k > kFusedMaxK)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize_select: k=%d must be a multiple of 16 in [16, min(cols, %d)]", k, kFusedMaxK);
  if ((scale_layout != QUADS_SCALES_LINEAR && scale_layout != QUADS_SCALES_TCGEN05) ||
      (r_scale_layout != QUADS_SCALES_LINEAR && r_scale_layout != QUADS_SCALES_TCGEN05))
    return fail(QUADS_ERR_INVALID_ARG, "quantize_select: bad scale layout");
  if (scale_layout == QUADS_SCALES_TCGEN05 && cols % 64)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize_select: TCGEN05 scale layout needs cols %% 64 == 0");
  if (ldx < cols || ldx % 8 || ld_codes < cols / 2 || ld_codes % 4 || !aligned16(x) ||
      !aligned16(codes))
    return fail(QUADS_ERR_MISALIGNED, "quantize_select: x and codes 16-byte aligned, ldx >= cols (%% 8), ld_codes >= cols/2 (%% 4)");
  const size_t need = quads_workspace_size(QUADS_OP_QUANTIZE_SELECT, rows, cols, 0, k, 1);
  if (rows > 0 && (!workspace || workspace_bytes < need))
    return fail(QUADS_ERR_WORKSPACE, "quantize_select: workspace needs %zu bytes", need);
  if (((uintptr_t)workspace | (uintptr_t)r_codes) & 15u)
    return fail(QUADS_ERR_MISALIGNED, "quantize_select: workspace and r_codes must be 16-byte aligned");
  if (rows == 0) return QUADS_OK;
  const int kpad = quads_kpad(k);
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
  FusedCtl* ctl = (FusedCtl*)ws;
  float* partials = (float*)(ws + 256);
  float* scores = (float*)(ws + 256 + al((size_t)((rows + 31) / 32) * cols * 4));
  float* rs = (float*)((char*)scores + al((size_t)cols * 4));
  if (scores_out) scores = scores_out;
  cudaMemsetAsync(ctl, 0, sizeof(FusedCtl), st);
  if (scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
    const int64_t start = (rows / 128) * (cols / 64) * 512;
    cudaMemsetAsync(scales + start, 0, (size_t)(sf_tc_bytes(rows, cols) - start), st);
  }
  if (r_scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
    const int64_t start = (rows / 128) * (kpad / 64) * 512;
    cudaMemsetAsync(r_scales + start, 0, (size_t)(sf_tc_bytes(rows, kpad) - start), st);
  }
  auto kernel = cols <= 2048 ? quantize_select_kernel<8>
                : cols <= 4096 ? quantize_select_kernel<16>
                               : quantize_select_kernel<32>;
  // every block must be resident at once (grid-wide barriers): one per SM
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kFusedThreads, 0);
  if (e != cudaSuccess || per_sm < 1)
    return fail(QUADS_ERR_CUDA, "quantize_select: occupancy query: %s", cudaGetErrorString(e));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeCooperative;
  at.val.cooperative = 1;
  // several small blocks per SM (the quantization phase needs the warps to
  // hide its load latency), all resident at once; no more blocks than
  // 32x256 quantization tasks, so that a small input (a decode batch) leaves
  // SMs to the work of other streams
  const int64_t ntasks = ((rows + 31) / 32) * ((cols + 255) / 256);
  const int64_t full = (int64_t)num_sms() * std::min(per_sm, 4);
  cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min(full, ntasks)), 1, 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, (const __nv_bfloat16*)x, rows, (int)cols, ldx, codes,
                         ld_codes, scales, (int)scale_layout, tensor_scale_out, partials,
                         scores, (int)k, kpad, sel, rs, r_codes, r_scales, (int)r_scale_layout,
                         r_tensor_scale, ctl, 2000000000ull);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(QUADS_ERR_CUDA, "quantize_select: cooperative launch: %s", cudaGetErrorString(e));
  }
  return check_launch("quantize_select", 1);
}

extern "C" quads_status_t quads_quantize_select_groups_nvfp4(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* group_offsets,
    int32_t num_groups, const int32_t* group_counts, const float* tensor_scale_in,
    const float* tensor_amax_in, int32_t k, uint8_t* codes, int64_t ld_codes, uint8_t* scales,
    int32_t scale_layout, float* tensor_scale_out, int32_t* sel, float* scores_out,
    uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout, float* r_tensor_scale,
    void* workspace, size_t workspace_bytes, void* sel_ready_event, void* stream) {
  if (rows > 0 && (!x || !group_offsets || !codes || !scales || !tensor_scale_out || !sel ||
                   !r_codes || !r_scales || !r_tensor_scale))
    return fail(QUADS_ERR_INVALID_ARG, "quantize_select_groups: null pointer argument");
  if (rows < 0 || cols < 16 || cols % 16 || cols > kQsgMaxCols)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize_select_groups: cols=%lld must be a multiple of 16 in [16, %d]", (long long)cols, kQsgMaxCols);
  if (k <= 0 || k % 16 || k > cols)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize_select_groups: k=%d must be a multiple of 16 in [16, cols]", k);
  if (num_groups < 1) return fail(QUADS_ERR_INVALID_ARG, "quantize_select_groups: num_groups < 1");
  if (tensor_scale_in && tensor_amax_in)
    return fail(QUADS_ERR_INVALID_ARG, "quantize_select_groups: give tensor_scale_in or tensor_amax_in, not both");
  if ((scale_layout != QUADS_SCALES_LINEAR && scale_layout != QUADS_SCALES_TCGEN05) ||
      (r_scale_layout != QUADS_SCALES_LINEAR && r_scale_layout != QUADS_SCALES_TCGEN05))
    return fail(QUADS_ERR_INVALID_ARG, "quantize_select_groups: bad scale layout");
  if (scale_layout == QUADS_SCALES_TCGEN05 && cols % 64)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize_select_groups: TCGEN05 scale layout needs cols %% 64 == 0");
  if (rows * (int64_t)k >= (1ll << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "quantize_select_groups: rows * k must be below 2^31");
  if (ldx < cols || ldx % 8 || ld_codes < cols / 2 || ld_codes % 4 || !aligned16(x) ||
      !aligned16(codes))
    return fail(QUADS_ERR_MISALIGNED, "quantize_select_groups: x and codes 16-byte aligned, ldx >= cols (%% 8), ld_codes >= cols/2 (%% 4)");
  const size_t need = quads_workspace_size(QUADS_OP_QUANTIZE_SELECT_GROUPS, rows, cols, 0, k,
                                           num_groups);
  if (rows > 0 && (!workspace || workspace_bytes < need))
    return fail(QUADS_ERR_WORKSPACE, "quantize_select_groups: workspace needs %zu bytes", need);
  if (((uintptr_t)workspace | (uintptr_t)r_codes) & 15u)
    return fail(QUADS_ERR_MISALIGNED, "quantize_select_groups: workspace and r_codes must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  auto sel_ready = [&]() -> quads_status_t {
    if (!sel_ready_event) return QUADS_OK;
    const cudaError_t e = cudaEventRecord((cudaEvent_t)sel_ready_event, st);
    return e == cudaSuccess ? QUADS_OK
                            : fail(QUADS_ERR_CUDA, "quantize_select_groups: cudaEventRecord: %s", cudaGetErrorString(e));
  };
  if (rows == 0) return sel_ready();
  const int kpad = quads_kpad(k);
  // the parts of the TCGEN05 scale arrays past the last full 128-row block
  // that no row covers read as zero
  if (scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
    const int64_t start = (rows / 128) * (cols / 64) * 512;
    cudaMemsetAsync(scales + start, 0, (size_t)(sf_tc_bytes(rows, cols) - start), st);
  }
  if (r_scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
    const int64_t start = (rows / 128) * (kpad / 64) * 512;
    cudaMemsetAsync(r_scales + start, 0, (size_t)(sf_tc_bytes(rows, kpad) - start), st);
  }
  // shared memory: the chunk's squares, then as many rows (bf16 values and
  // scale bytes) as fit what is left -- groups of up to that many real rows
  // keep them on chip for R_sel
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa = {};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, quantize_select_groups_kernel);
  if (e != cudaSuccess)
    return fail(QUADS_ERR_CUDA, "quantize_select_groups: attribute query: %s", cudaGetErrorString(e));
  const size_t sq_bytes = (size_t)kScoreChunk * cols * 4;
  const int64_t left = (int64_t)optin - (int64_t)fa.sharedSizeBytes - (int64_t)sq_bytes - 1024;
  const int stash_rows = (int)std::max<int64_t>(0, std::min<int64_t>(256, left / (cols * 2 + cols / 16)));
  const size_t smem = sq_bytes + (size_t)stash_rows * (cols * 2 + cols / 16);
  e = cudaFuncSetAttribute(quantize_select_groups_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess)
    return fail(QUADS_ERR_CUDA, "quantize_select_groups: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  // one block per group, plus blocks that zero the R_sel rows past the last group
  launch_dep(quantize_select_groups_kernel, num_groups + 32, kQsgThreads, smem, st,
      (const __nv_bfloat16*)x, rows, (int)cols, ldx, group_offsets, (int)num_groups, group_counts,
      tensor_scale_in, tensor_amax_in, codes, ld_codes, scales, (int)scale_layout,
      tensor_scale_out, (int)k, kpad, sel, scores_out, (float*)workspace, r_codes, r_scales,
      (int)r_scale_layout, r_tensor_scale, stash_rows);
  if (quads_status_t s = check_launch("quantize_select_groups", 1)) return s;
  return sel_ready();
}

extern "C" quads_status_t quads_trace_round(const void* x_train, int64_t rows, int64_t cols,
                                            int64_t ldx, const uint8_t* rollout_codes,
                                            int64_t ld_codes, const uint8_t* rollout_scales,
                                            const float* rollout_tensor_scale, uint8_t* codes_out,
                                            unsigned long long* counters, void* stream) {
  if (rows > 0 && (!x_train || !rollout_codes || !rollout_scales || !rollout_tensor_scale || !codes_out))
    return fail(QUADS_ERR_INVALID_ARG, "trace_round: null pointer argument");
  if (cols <= 0 || cols % 16) return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_round: cols %% 16");
  if (ldx < cols || ldx % 8 || ld_codes < cols / 2 || ld_codes % 4 || !aligned16(x_train) ||
      ((uintptr_t)rollout_codes & 3u) || ((uintptr_t)codes_out & 3u))
    return fail(QUADS_ERR_MISALIGNED, "trace_round: leading dimensions / alignment");
  if (rows == 0) return QUADS_OK;
  if (rows * (cols / 8) >= ((int64_t)1 << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_round: rows * cols / 8 must be < 2^31");
  cudaStream_t st = (cudaStream_t)stream;
  trace_kernel<false><<<grid_for(rows * (cols / 16), 256), 256, 0, st>>>(
      (const __nv_bfloat16*)x_train, rows, (int)cols, ldx, rollout_codes, ld_codes,
      rollout_scales, rollout_tensor_scale, codes_out, counters);
  return check_launch("trace_round", 1);
}

extern "C" quads_status_t quads_trace_round_mx(const void* x_train, int64_t rows, int64_t cols,
                                               int64_t ldx, const uint8_t* rollout_codes,
                                               int64_t ld_codes, const uint8_t* rollout_scales,
                                               uint8_t* codes_out, unsigned long long* counters,
                                               void* stream) {
  if (rows > 0 && (!x_train || !rollout_codes || !rollout_scales || !codes_out))
    return fail(QUADS_ERR_INVALID_ARG, "trace_round_mx: null pointer argument");
  if (cols <= 0 || cols % 32) return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_round_mx: cols %% 32");
  if (ldx < cols || ldx % 8 || ld_codes < cols / 2 || ld_codes % 4 || !aligned16(x_train) ||
      ((uintptr_t)rollout_codes & 3u) || ((uintptr_t)codes_out & 3u))
    return fail(QUADS_ERR_MISALIGNED, "trace_round_mx: leading dimensions / alignment");
  if (rows < 0 || rows * (cols / 8) >= ((int64_t)1 << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_round_mx: rows * cols / 8 must be < 2^31");
  if (rows == 0) return QUADS_OK;
  trace_kernel<true><<<grid_for(rows * (cols / 16), 256), 256, 0, (cudaStream_t)stream>>>(
      (const __nv_bfloat16*)x_train, rows, (int)cols, ldx, rollout_codes, ld_codes,
      rollout_scales, nullptr, codes_out, counters);
  return check_launch("trace_round_mx", 1);
}

extern "C" quads_status_t quads_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                            uint8_t* codes, int64_t ld_codes, uint8_t* scales,
                                            int32_t scale_layout, void* y_qdq, int64_t ldy,
                                            void* stream) {
  if (rows > 0 && (!x || !codes || !scales))
    return fail(QUADS_ERR_INVALID_ARG, "mx_quantize: null x/codes/scales");
  if (rows < 0 || cols <= 0 || cols % 32)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "mx_quantize: cols %% 32 == 0");
  if (scale_layout != QUADS_SCALES_LINEAR && scale_layout != QUADS_SCALES_TCGEN05)
    return fail(QUADS_ERR_INVALID_ARG, "mx_quantize: bad scale_layout %d", scale_layout);
  if (scale_layout == QUADS_SCALES_TCGEN05 && cols % 128)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "mx_quantize: TCGEN05 scale layout needs cols %% 128 == 0");
  if (ldx < cols || ldx % 8 || !aligned16(x) || ld_codes < cols / 2 || ld_codes % 8 ||
      ((uintptr_t)codes & 7u))
    return fail(QUADS_ERR_MISALIGNED, "mx_quantize: x 16-byte aligned (ldx >= cols, %% 8), codes 8-byte aligned (ld_codes >= cols/2, %% 8)");
  if (y_qdq && (ldy < cols || ldy % 8 || !aligned16(y_qdq)))
    return fail(QUADS_ERR_MISALIGNED, "mx_quantize: y 16-byte aligned, ldy >= cols, %% 8");
  if (rows * (cols / 16) >= ((int64_t)1 << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "mx_quantize: rows * cols / 16 must be < 2^31");
  if (rows == 0) return QUADS_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (scale_layout == QUADS_SCALES_TCGEN05 && rows % 128) {
    const int64_t start = (rows / 128) * (cols / 128) * 512;
    const int64_t bytes = ((rows + 127) / 128) * 128 * (cols / 32);
    cudaMemsetAsync(scales + start, 0, (size_t)(bytes - start), st);
  }
  mx_quantize_kernel<<<grid_for(rows * (cols / 16), 256), 256, 0, st>>>(
      (const __nv_bfloat16*)x, rows, (int)cols, ldx, codes, ld_codes, scales, scale_layout,
      (__nv_bfloat16*)y_qdq, ldy);
  return check_launch("mx_quantize", 1);
}

extern "C" quads_status_t quads_trace_pack_record(const uint8_t* rollout_codes, int64_t rows,
                                                  int64_t cols, int64_t ld_codes,
                                                  uint8_t* mantissa_bits, int64_t ld_bits,
                                                  void* stream) {
  if (rows > 0 && (!rollout_codes || !mantissa_bits))
    return fail(QUADS_ERR_INVALID_ARG, "trace_pack_record: null pointer argument");
  if (rows < 0 || cols <= 0 || cols % 16 || ld_codes < cols / 2 || ld_codes % 4 ||
      ld_bits < cols / 8)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_pack_record: cols %% 16, ld_codes >= cols/2 (%% 4), ld_bits >= cols/8");
  if (((uintptr_t)rollout_codes & 3u) != 0)
    return fail(QUADS_ERR_MISALIGNED, "trace_pack_record: rollout_codes must be 4-byte aligned");
  if (rows * (cols / 8) >= ((int64_t)1 << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_pack_record: rows * cols / 8 must be < 2^31");
  if (rows == 0) return QUADS_OK;
  // 32 codes per thread when rows are 16-byte aligned runs of codes and the
  // record rows take aligned 4-byte stores
  const int vec = cols % 32 == 0 && ld_codes % 16 == 0 && ld_bits % 4 == 0 &&
                  ((uintptr_t)rollout_codes & 15) == 0 && ((uintptr_t)mantissa_bits & 3) == 0;
  trace_pack_kernel<<<grid_for(rows * (cols / (vec ? 32 : 8)), 256), 256, 0, (cudaStream_t)stream>>>(
      rollout_codes, rows, (int)cols, ld_codes, mantissa_bits, ld_bits, vec);
  return check_launch("trace_pack_record", 1);
}

extern "C" quads_status_t quads_trace_round_1bit(const void* x_train, int64_t rows, int64_t cols,
                                                 int64_t ldx, const uint8_t* mantissa_bits,
                                                 int64_t ld_bits, const uint8_t* rollout_scales,
                                                 const float* rollout_tensor_scale,
                                                 uint8_t* codes_out, int64_t ld_codes,
                                                 unsigned long long* counters, void* stream) {
  if (rows > 0 && (!x_train || !mantissa_bits || !rollout_scales || !rollout_tensor_scale || !codes_out))
    return fail(QUADS_ERR_INVALID_ARG, "trace_round_1bit: null pointer argument");
  if (rows < 0 || cols <= 0 || cols % 16 || ld_bits < cols / 8 || ld_codes < cols / 2 ||
      ld_codes % 4)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_round_1bit: cols %% 16, ld_bits >= cols/8, ld_codes >= cols/2 (%% 4)");
  if (ldx < cols || ldx % 8 || !aligned16(x_train) || ((uintptr_t)codes_out & 3u) != 0)
    return fail(QUADS_ERR_MISALIGNED, "trace_round_1bit: x_train 16-byte aligned (ldx >= cols, %% 8), codes_out 4-byte aligned");
  if (rows * (cols / 8) >= ((int64_t)1 << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "trace_round_1bit: rows * cols / 8 must be < 2^31");
  if (rows == 0) return QUADS_OK;
  trace_1bit_kernel<<<grid_for(rows * (cols / 16), 256), 256, 0, (cudaStream_t)stream>>>(
      (const __nv_bfloat16*)x_train, rows, (int)cols, ldx, mantissa_bits, ld_bits,
      rollout_scales, rollout_tensor_scale, codes_out, ld_codes, counters);
  return check_launch("trace_round_1bit", 1);
}
