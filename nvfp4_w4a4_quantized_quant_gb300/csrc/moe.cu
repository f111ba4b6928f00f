// MoE dispatch around the grouped compensated GEMM: router top-k with gate
// weights, the deterministic token -> expert row plan (groups padded to 128
// rows), the gather of NVFP4 rows into expert order, and the gate-weighted
// combine.  [TRACE digest] "MoE 专家路由敏感性": the router sends every token to a
// few experts by gate score.
//
// Determinism: counts and row positions are prefix counts over tokens (no
// atomics), so the plan is identical from run to run.
#include <algorithm>
#include <cstdio>

#include "common.cuh"

namespace quads {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 16;

constexpr int kRouteTokens = 32;   // tokens per routing block: one warp each

// One block of 32 warps per 32 consecutive tokens, one warp per token.  Lane l
// holds logits l, l+32, ...; round r takes the warp arg-max (ties -> lower
// expert id), removes it, and lane r keeps it.  The chosen experts are ranked
// by id (ascending slot order) and gates are exp(l - lmax) / sum over the
// chosen.  Then, from the block's per-token expert bit masks in shared
// memory: each (token, slot) gets its rank among the block's earlier tokens
// routed to the same expert (stored in token_row, turned into a row by
// assign_kernel), and each expert its count of the block's tokens, written to
// bcount[e][block] -- no atomics, so every number is independent of
// scheduling.
// W: 32-expert words held per lane (the smallest power of two >= E / 32), so
// an arg-max round scans only the lanes' real expert slots; two 1024-thread
// blocks per SM (32 registers), so that the token blocks of a large batch are
// resident in one wave.
template <int W>
__global__ void __launch_bounds__(1024, 2) route_kernel(const float* __restrict__ logits, int T,
                                                     int E, int topk, int32_t* __restrict__ idx,
                                                     float* __restrict__ gates,
                                                     int32_t* __restrict__ bcount,
                                                     int32_t* __restrict__ local_rank) {
  griddep_wait();
  __shared__ uint32_t smask[kRouteTokens][kMaxExperts / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kRouteTokens + warp;
  const int words = (E + 31) >> 5;
  const bool live = t < T;
  int my_e = 0x7fffffff, rank = 0;
  if (live) {
    float v[W];
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const int e = lane + 32 * i;
      const float l = (i < words && e < E) ? logits[(int64_t)t * E + e] : -INFINITY;
      v[i] = isnan(l) ? -INFINITY : l;   // a NaN logit ranks lowest: every pick is a real expert
    }
    uint32_t taken = 0;
    float my_l = -INFINITY, lmax = -INFINITY;
    for (int r = 0; r < topk; ++r) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < W; ++i) {
        const int e = lane + 32 * i;
        if (i < words && e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      if (r == 0) lmax = bv;
      if (lane == r) { my_e = be; my_l = bv; }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
    }
    const bool mine = lane < topk;
    float p = mine ? expf(my_l - lmax) : 0.0f;
    float s = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    for (int j = 0; j < topk; ++j) {
      const int ej = __shfl_sync(0xffffffffu, my_e, j);
      rank += (ej < my_e) ? 1 : 0;
    }
    if (mine) {
      idx[(int64_t)t * topk + rank] = my_e;
      gates[(int64_t)t * topk + rank] = p / s;
    }
    for (int w = 0; w < words; ++w) {
      const uint32_t bit = (mine && (my_e >> 5) == w) ? (1u << (my_e & 31)) : 0u;
      const uint32_t m = __reduce_or_sync(0xffffffffu, bit);
      if (lane == 0) smask[warp][w] = m;
    }
  }
  __syncthreads();
  const int nlive = min(kRouteTokens, T - (int)blockIdx.x * kRouteTokens);
  if (live && lane < topk) {
    const int mw = my_e >> 5;
    const uint32_t mb = 1u << (my_e & 31);
    int r = 0;
    for (int i = 0; i < warp; ++i) r += (smask[i][mw] & mb) ? 1 : 0;
    local_rank[(int64_t)t * topk + rank] = r;
  }
  if ((int)threadIdx.x < E) {
    const int mw = threadIdx.x >> 5;
    const uint32_t mb = 1u << (threadIdx.x & 31);
    int c = 0;
    for (int i = 0; i < nlive; ++i) c += (smask[i][mw] & mb) ? 1 : 0;
    bcount[(int64_t)threadIdx.x * gridDim.x + blockIdx.x] = c;
  }
}

// One block per expert: block_prefix[e][b] = tokens of expert e in routing
// blocks < b and the expert's total count, by a block-wide scan (thread t
// takes 8 consecutive routing blocks per pass).  The padded offsets are formed
// by assign_kernel from the counts.
__global__ void __launch_bounds__(256) plan_kernel(const int32_t* __restrict__ bcount, int nb,
                                                   int32_t* __restrict__ bprefix,
                                                   int32_t* __restrict__ counts) {
  griddep_wait();
  __shared__ int warp_sums[8];
  const int e = blockIdx.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int32_t* bc = bcount + (int64_t)e * nb;
  int32_t* bp = bprefix + (int64_t)e * nb;
  int running = 0;
  for (int b0 = 0; b0 < nb; b0 += 256 * 8) {
    int v[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int b = b0 + 8 * (int)threadIdx.x + i;
      v[i] = b < nb ? bc[b] : 0;
      sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    int before = running, total = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      total += warp_sums[i];
      if (i < w) before += warp_sums[i];
    }
    int x = before + incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int b = b0 + 8 * (int)threadIdx.x + i;
      if (b < nb) bp[b] = x;
      x += v[i];
    }
    running += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) counts[e] = running;
}

// Rows of the plan: slot (t, j) routed to expert e goes to row
// off[e] + block_prefix[e][t / 32] + its rank within the routing block, so
// each expert's rows hold its tokens in ascending token order.  Padding rows
// get row_token = -1.  Every block forms the padded offsets
// off[e+1] = off[e] + roundup(count[e], 128) itself (a scan over <= 256
// experts); block 0 stores them.
__global__ void __launch_bounds__(256) assign_kernel(const int32_t* __restrict__ idx, int T, int E,
                                                     int topk, int nb,
                                                     const int32_t* __restrict__ bprefix,
                                                     int32_t* __restrict__ off_out,
                                                     const int32_t* __restrict__ counts,
                                                     int32_t* __restrict__ row_token,
                                                     int32_t* __restrict__ token_row,
                                                     int64_t cap) {
  griddep_wait();
  __shared__ int off[kMaxExperts + 1];
  __shared__ int warp_sums[8];
  {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = (int)threadIdx.x < E ? counts[threadIdx.x] : 0;
    const int pc = (c + QUADS_MOE_ROW_ALIGN - 1) / QUADS_MOE_ROW_ALIGN * QUADS_MOE_ROW_ALIGN;
    int incl = pc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < w; ++i) before += warp_sums[i];
    if ((int)threadIdx.x < E) off[threadIdx.x + 1] = before + incl;
    if (threadIdx.x == 0) off[0] = 0;
    __syncthreads();
    // E + 1 offsets (257 with 256 experts: more than the block's threads)
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i <= E; i += blockDim.x) off_out[i] = off[i];
  }
  const int total = T * topk;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int t = i / topk;
    const int e = idx[i];
    if (!QDBG(e >= 0 && e < E)) continue;
    const int row = off[e] + bprefix[(int64_t)e * nb + t / kRouteTokens] + token_row[i];
    token_row[i] = row;
    if (QDBG(row >= 0 && row < cap)) row_token[row] = t;
  }
  for (int e = blockIdx.x; e < E; e += gridDim.x)
    for (int r = off[e] + counts[e] + (int)threadIdx.x; r < off[e + 1]; r += blockDim.x)
      if (QDBG(r < cap)) row_token[r] = -1;
}

// Wide rows (>= 32 code vectors of 16 bytes): a warp copies 4 rows at a time,
// lane = vector, all loads issued before the stores; then the scales in a
// second pass over (128-row block, 4-column group) items: in the TCGEN05
// layout the 16 bytes at lane l of an atom hold rows l, l+32, l+64 and l+96
// of the block, so lane l gathers those four rows' 4-byte groups and stores
// them as one 16-byte word -- a warp writes the atom's 512 bytes whole
// (4-byte stores at a 512-byte stride left most of each sector to be merged
// in L2); a block that reaches past the last row keeps 4-byte stores for its
// rows.  Narrow rows (the k-channel residual slices): one pass over a thread
// per (row, vector) and a thread per (128-row block, scale group, lane) with
// the same whole-word scale stores, 32-bit index math.  Padding rows
// (row_token -1) get zero codes and scales.
__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ row_token,
                                                     const int32_t* __restrict__ off, int E,
                                                     int64_t cap, int cols,
                                                     const uint8_t* __restrict__ ic,
                                                     const uint8_t* __restrict__ isf,
                                                     uint8_t* __restrict__ oc,
                                                     uint8_t* __restrict__ osf) {
  griddep_wait();
  int64_t nrows = off[E];
  if (!QDBG(nrows >= 0 && nrows <= cap)) nrows = 0;
  const int cbytes = cols >> 1;
  const int ncols16 = cols >> 4;
  const int nvec = cbytes >> 4;           // 16-byte vectors per row
  const int natom = ncols16 >> 2;         // 4-byte scale groups per row
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = nthreads >> 5;
  if (nvec >= 32) {
    for (int64_t r0 = (tid >> 5) * 4; r0 < nrows; r0 += nwarps * 4) {
      int t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) t[u] = r0 + u < nrows ? __ldg(row_token + r0 + u) : -2;
      for (int v0 = lane; v0 < nvec; v0 += 64) {
        uint4 buf[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int v = v0 + 32 * h;
            buf[u][h] = make_uint4(0, 0, 0, 0);
            if (t[u] >= 0 && v < nvec && QDBG(t[u] < (1 << 30)))
              buf[u][h] = __ldg(reinterpret_cast<const uint4*>(ic + (int64_t)t[u] * cbytes) + v);
          }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int v = v0 + 32 * h;
            if (t[u] != -2 && v < nvec)
              reinterpret_cast<uint4*>(oc + (r0 + u) * cbytes)[v] = buf[u][h];
          }
      }
    }
  } else {
    // narrow rows: nvec < 32, natom < 8; rows * nvec fits comfortably in 32
    // bits.  Codes and the 4-byte scale groups in one pass (one round trip
    // for the small residual slices, where latency decides)
    // scale items: (128-row block, 4-column group, lane l) -> rows l, l+32,
    // l+64, l+96 of the block, one 16-byte store (32 lanes: a whole atom)
    const uint32_t ncode = (uint32_t)(nrows * nvec);
    const uint32_t nsc = (uint32_t)(((nrows + 127) >> 7) * natom * 32);
    for (uint32_t i = (uint32_t)tid; i < ncode + nsc; i += (uint32_t)nthreads) {
      if (i < ncode) {
        const uint32_t r = i / (uint32_t)nvec, v = i - r * (uint32_t)nvec;
        const int t = __ldg(row_token + r);
        uint4 x = make_uint4(0, 0, 0, 0);
        if (t >= 0) x = __ldg(reinterpret_cast<const uint4*>(ic + (int64_t)t * cbytes) + v);
        reinterpret_cast<uint4*>(oc)[i] = x;
      } else {
        const uint32_t j = i - ncode;
        const uint32_t item = j >> 5, l = j & 31u;
        const uint32_t rb = item / (uint32_t)natom, a = item - rb * (uint32_t)natom;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t r = (int64_t)rb * 128 + l + 32 * q;
          const int t = r < nrows ? __ldg(row_token + r) : -1;
          w[q] = t >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(isf + (int64_t)t * ncols16) + a) : 0u;
        }
        uint8_t* atom = osf + ((int64_t)rb * natom + a) * 512 + l * 16;
        if ((int64_t)rb * 128 + 128 <= nrows) {
          *reinterpret_cast<uint4*>(atom) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if ((int64_t)rb * 128 + l + 32 * q < nrows) *reinterpret_cast<uint32_t*>(atom + q * 4) = w[q];
        }
      }
    }
    return;
  }
  // wide rows' scales: a warp per (128-row block, 4-column group)
  const int64_t nblk = (nrows + 127) >> 7;
  for (int64_t item = tid >> 5; item < nblk * natom; item += nwarps) {
    const int64_t rb = item / natom;
    const int a = (int)(item - rb * natom);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t r = rb * 128 + lane + 32 * q;
      const int t = r < nrows ? __ldg(row_token + r) : -1;
      w[q] = t >= 0 && QDBG(t < (1 << 30))
                 ? __ldg(reinterpret_cast<const uint32_t*>(isf + (int64_t)t * ncols16) + a)
                 : 0u;
    }
    uint8_t* atom = osf + (rb * natom + a) * 512;
    if (rb * 128 + 128 <= nrows) {
      *reinterpret_cast<uint4*>(atom + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (rb * 128 + lane + 32 * q < nrows)
          *reinterpret_cast<uint32_t*>(atom + lane * 16 + q * 4) = w[q];
    }
  }
}

// out[t, :] = bf16(sum_j gate[t, j] * y[row(t, j), :]), float32, j ascending.
// kTopk > 0: the slot count is known at compile time, so every slot's row
// index and then every slot's y vector are loaded before the sum (kTopk
// loads in flight per thread); the sum itself keeps the same order.
template <int kTopk>
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                      int64_t ldy,
                                                      const int32_t* __restrict__ token_row,
                                                      const float* __restrict__ gates, int T,
                                                      int topk, int H, __nv_bfloat16* __restrict__ out,
                                                      int64_t ldo) {
  griddep_wait();
  const int vec = H >> 3;
  const int64_t total = (int64_t)T * vec;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / vec);
    const int c = (int)(i % vec) * 8;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (kTopk > 0) {
      int r[kTopk > 0 ? kTopk : 1];
      float g[kTopk > 0 ? kTopk : 1];
      uint4 v[kTopk > 0 ? kTopk : 1];
#pragma unroll
      for (int j = 0; j < kTopk; ++j) {
        r[j] = token_row[(int64_t)t * kTopk + j];
        g[j] = gates[(int64_t)t * kTopk + j];
      }
#pragma unroll
      for (int j = 0; j < kTopk; ++j)
        v[j] = QDBG(r[j] >= 0) ? *reinterpret_cast<const uint4*>(y + (int64_t)r[j] * ldy + c)
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < kTopk; ++j) {
        float f[8];
        bf16x8_to_f32(v[j], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(g[j], f[q], acc[q]);
      }
    } else {
      for (int j = 0; j < topk; ++j) {
        const int r = token_row[(int64_t)t * topk + j];
        const float g = gates[(int64_t)t * topk + j];
        float f[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(y + (int64_t)r * ldy + c), f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, f[q], acc[q]);
      }
    }
    uint32_t pk[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      pk[q] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(out + (int64_t)t * ldo + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

int debug_line_moe(long long* value) { return take_debug_line(value); }

}  // namespace quads

using namespace quads;

extern "C" quads_status_t quads_moe_route(const float* logits, int32_t tokens, int32_t num_experts,
                                          int32_t topk, int32_t* topk_idx, float* gates,
                                          int32_t* expert_counts, int32_t* expert_offsets,
                                          int32_t* row_token, int32_t* token_row,
                                          int64_t rows_capacity, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (!expert_counts || !expert_offsets || !row_token ||
      (tokens > 0 && (!logits || !topk_idx || !gates || !token_row)))
    return fail(QUADS_ERR_INVALID_ARG, "moe_route: null pointer argument");
  if (tokens < 0 || num_experts < 1 || num_experts > kMaxExperts || topk < 1 ||
      topk > kMaxTopk || topk > num_experts)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "moe_route: need 1<=experts<=256, 1<=topk<=min(16, experts)");
  if (rows_capacity < (int64_t)tokens * topk + (int64_t)num_experts * (QUADS_MOE_ROW_ALIGN - 1))
    return fail(QUADS_ERR_INVALID_ARG, "moe_route: rows_capacity too small");
  const size_t need = quads_workspace_size(QUADS_OP_MOE_ROUTE, tokens, num_experts, 0, topk, 1);
  if (!workspace || workspace_bytes < need)
    return fail(QUADS_ERR_WORKSPACE, "moe_route: workspace needs %zu bytes", need);
  if ((uintptr_t)workspace & 15u) return fail(QUADS_ERR_MISALIGNED, "moe_route: workspace must be 16-byte aligned");
  const int nb = (tokens + kRouteTokens - 1) / kRouteTokens;
  int32_t* bcount = (int32_t*)workspace;                       // [E, nb]
  int32_t* bprefix = bcount + (size_t)nb * num_experts;         // [E, nb]
  cudaStream_t st = (cudaStream_t)stream;
  if (tokens > 0)
    {
      const int words = (num_experts + 31) / 32;
      auto rk = words <= 1 ? route_kernel<1> : words <= 2 ? route_kernel<2>
              : words <= 4 ? route_kernel<4> : route_kernel<8>;
      launch_dep(rk, nb, 32 * kRouteTokens, 0, st,
          logits, tokens, num_experts, topk, topk_idx, gates, bcount, token_row);
    }
  launch_dep(plan_kernel, num_experts, 256, 0, st, bcount, nb, bprefix, expert_counts);
  const int assign_blocks = std::max(1, std::min(num_sms() * 4, (tokens * topk + 255) / 256));
  launch_dep(assign_kernel, assign_blocks, 256, 0, st, topk_idx, tokens, num_experts, topk, nb,
             bprefix, expert_offsets, expert_counts, row_token, token_row, rows_capacity);
  return check_launch("moe_route", tokens > 0 ? 3 : 2);
}

extern "C" quads_status_t quads_moe_gather(const int32_t* row_token, const int32_t* expert_offsets,
                                           int32_t num_experts, int64_t rows_capacity,
                                           int64_t cols, const uint8_t* in_codes,
                                           const uint8_t* in_scales, uint8_t* out_codes,
                                           uint8_t* out_scales, void* stream) {
  if (!row_token || !expert_offsets || !in_codes || !in_scales || !out_codes || !out_scales)
    return fail(QUADS_ERR_INVALID_ARG, "moe_gather: null pointer argument");
  if (cols <= 0 || cols % 64 || rows_capacity % 128)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "moe_gather: cols %% 64 and rows_capacity %% 128");
  // output scales go out as whole 16-byte atom words
  if (((uintptr_t)in_codes | (uintptr_t)out_codes | (uintptr_t)out_scales) & 15u || (uintptr_t)in_scales & 3u)
    return fail(QUADS_ERR_MISALIGNED, "moe_gather: codes and out_scales 16-byte, in_scales 4-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  if (cols / 32 < 32 && rows_capacity * (cols / 32 + cols / 64) >= (int64_t)1 << 31)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "moe_gather: narrow rows need rows * cols / 32 < 2^31");
  const int64_t vecs = rows_capacity * (cols / 32);   // 16-byte code vectors
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((vecs / 4 + 255) / 256, (int64_t)num_sms() * 8));
  launch_dep(gather_kernel, blocks, 256, 0, st,
      row_token, expert_offsets, num_experts, rows_capacity, (int)cols, in_codes, in_scales,
      out_codes, out_scales);
  return check_launch("moe_gather", 1);
}

extern "C" quads_status_t quads_moe_combine(const void* y, int64_t ldy, const int32_t* token_row,
                                            const float* gates, int32_t tokens, int32_t topk,
                                            int64_t hidden, void* out, int64_t ldo, void* stream) {
  if (tokens > 0 && (!y || !token_row || !gates || !out))
    return fail(QUADS_ERR_INVALID_ARG, "moe_combine: null pointer");
  if (hidden <= 0 || hidden % 8 || ldy % 8 || ldo % 8 || ldy < hidden || ldo < hidden)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "moe_combine: hidden/ld must be multiples of 8");
  if (((uintptr_t)y | (uintptr_t)out) & 15u)
    return fail(QUADS_ERR_MISALIGNED, "moe_combine: y and out must be 16-byte aligned");
  if (tokens == 0) return QUADS_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t work = (int64_t)tokens * (hidden / 8);
  const int blocks = (int)std::min<int64_t>((work + 255) / 256, (int64_t)num_sms() * 8);
  auto kernel = topk == 8   ? combine_kernel<8>
                : topk == 4 ? combine_kernel<4>
                : topk == 2 ? combine_kernel<2>
                : topk == 1 ? combine_kernel<1>
                            : combine_kernel<0>;
  launch_dep(kernel, blocks, 256, 0, st,
      (const __nv_bfloat16*)y, ldy, token_row, gates, tokens, topk, (int)hidden,
      (__nv_bfloat16*)out, ldo);
  return check_launch("moe_combine", 1);
}
