// Compensated NVFP4 W4A4 GEMM on the sm_103a tensor cores.
//
//   Y = s_a s_w * Q(A) Q(W)^T  +  s_r s_w * Q(R_sel) Q(W_sel)^T
//
// [QUADS technical summary] 2.2 B "Mechanism": the correction of the selected
// high-residual channels is added back to the quantized output; section 1: the
// bulk stays a native W4A4 GEMM.  Here both products run in one persistent
// kernel: the main K loop accumulates into one TMEM accumulator, the k-channel
// correction loop into a second one, and the epilogue forms a1*acc1 + a2*acc2.
//
// Design (one CTA per SM, 128x128 output tiles, K tiles of 512 FP4 = 256 B):
//   warps 0-2   TMA producers: A/B code tiles by tensor-map TMA (128B
//               swizzle) and scale atoms by bulk copy into a 3-stage x 72 KB
//               smem ring; a 512-element K tile is eight 8 KB boxes (A and B,
//               two 128-byte sub-tiles of two 64-row halves each) and two 4 KB
//               atom runs, 24 KB per warp.  One issuing warp
//               moves only ~29 B/cycle into its SM (its copies are processed
//               one after another); three keep up with the ~70 B/cycle/SM
//               that L2 delivers when every SM is loading.
//   warp 3      TMEM allocator + MMA issuer.  The warp stays converged: all
//               lanes poll the barriers and run every tcgen05 instruction,
//               predicated inside the asm on an elect.sync lane (a branch on
//               the elected lane plus __syncwarp costs ~200 cycles a stage):
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=128, K=64).
//   warps 4-7   scale staging: once a stage has landed, each warp copies a
//               quarter of its scale atoms from smem into TMEM with tcgen05.cp
//               (issued from four warps because each copy holds its issuing
//               thread for ~100 cycles) and its tcgen05.commit tells the MMA
//               warp when they are in place.  Reading the atoms with
//               ld.shared instead stalls for ~1-7K cycles while the MMAs
//               stream their operands (they take the whole smem bandwidth),
//               and loading them from global memory exposes L2 latency.
//   warps 8-15  epilogue: tcgen05.ld of both accumulators, scale, store (one
//               32-byte store per 16 bf16 outputs of a row when the rows are
//               32-byte aligned); two warps per TMEM lane quadrant, each owning
//               half of the columns.
// MXFP4 operands (E8M0 scale per 32 elements, no tensor scales) run through the
// same kernel with kind::mxf4 MMAs and one scale atom per two K steps.
// TMEM columns: acc1 double-buffered (0-127, 128-255), acc2 (256-383),
// scale-factor ring (384-511, 2 buffers x 64 columns).
// Every mbarrier wait is bounded (2 s); on a timeout the kernel latches an
// error word and every role stops.  Each producer warp then waits a fixed
// bounded time (200 us) for its copies in flight, the MMA and scale warps
// commit and wait (bounded) for their tensor-core work, and TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace quads {
namespace gemm {

constexpr int BM = 128, BN = 128;
constexpr int KSUB = 128;                     // bytes per row of one 128B-swizzled sub-tile (256 FP4)
constexpr int A_SUB = BM * KSUB;              // 16 KB
constexpr int B_SUB = BN * KSUB;              // 16 KB
constexpr int BOX_ROWS = 64;                  // rows per TMA box: half a 128-row sub-tile
constexpr int BOX_BYTES = BOX_ROWS * KSUB;    // 8 KB
constexpr int PRODUCERS = 3;
constexpr int NUM_THREADS = 512;  // 16 warps: 3 producers, MMA, 4 scale staging, 8 epilogue
constexpr int EPI_THREADS = 256;
constexpr int SF_WARPS = 4;
constexpr int MMA_WARP = 3, SF_WARP0 = 4, EPI_WARP0 = 8;
constexpr int TMEM_COLS = 512;
constexpr int ACC2_COL = 256;
constexpr int SF_COL = 384;
constexpr int MAX_GROUPS = 256;                 // experts cached in shared memory
constexpr int META_BYTES = 1024 + 4 * (MAX_GROUPS + 1) + 4 * 4 * MAX_GROUPS;
constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per wait

// Stage geometry of the 128x128-tile kernel: KS 256-element sub-tiles per
// stage, NS ring stages, NSF TMEM scale buffers.  Two are instantiated: 512-
// element stages (three of 72 KB, two scale buffers) and 256-element stages
// (six of 36 KB, four buffers), the latter for K not a multiple of 512, where
// a 512-element ring would carry half-empty stages (K = 768: 158 -> 144 us
// for the compensated GEMM2 shape; K = 2048 runs faster on 512).
template <int KS, int NS, int NSF>
struct Geo {
  static constexpr int KSUBS = KS;                     // sub-tiles per stage
  static constexpr int KSTEPS = 4 * KS;                // K=64 MMA steps per stage
  static constexpr int KTILE = 256 * KS;               // FP4 elements per stage
  static constexpr int STAGES = NS;
  static constexpr int A_TILE = A_SUB * KS;
  static constexpr int B_TILE = B_SUB * KS;
  static constexpr int SF_TILE = KSTEPS * 512;         // scale atoms (128 rows x 4 blocks each) per operand
  static constexpr int STAGE_BYTES = A_TILE + B_TILE + 2 * SF_TILE;
  static constexpr int BOXES = 2 * KS * 2;             // per stage: (A, B) x sub-tiles x halves
  static constexpr int COPIES = BOXES + 2;             // + the SFA and SFB atom runs (bulk copies)
  static constexpr int SF_BUFS = NSF;                  // TMEM scale buffers
  static constexpr int SF_BUF_COLS = 2 * 4 * KSTEPS;   // SFA and SFB: four columns per K step each
  static constexpr int SMEM_BYTES = NS * STAGE_BYTES + META_BYTES + 1024 /*align*/;
  static_assert(NSF * SF_BUF_COLS <= 128, "scale buffers fit the 128 TMEM columns left");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  // the stage's copies dealt to the producer warps: warp w issues [first, first + count)
  __host__ __device__ static constexpr int copies_first(int w) { return w * COPIES / PRODUCERS; }
};
using Geo512 = Geo<2, 3, 2>;
using Geo256 = Geo<1, 6, 4>;

enum { OUT_F32 = 0, OUT_BF16 = 1, OUT_SWIGLU = 2 };

struct Params {
  int E, N, K, kpad, Nt;
  int64_t M;                    // dense rows (row_off == nullptr)
  const int32_t* row_off;       // [E+1] padded row offsets (multiples of 128) or null
  const int32_t* row_cnt;       // [E] real rows (null: all rows of the tile range are real)
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const uint8_t* r_sf;
  const uint8_t* ws_sf;
  const float* a_ts;
  const float* b_ts;
  const float* r_ts;
  int a_ts_pe, r_ts_pe;
  int comp;
  int mx;                       // MXFP4 operands: E8M0 scale per 32 elements, no tensor scales
  void* y;
  int64_t ldy;
  int out_mode;
  int st32;                     // y rows and base 32-byte aligned: one 32-byte store per 16 bf16
  uint32_t* y_amax;             // nullable [E]: max |stored y| per group (float bits)
  int* err;
  // extents for the bounds-checked build: scale buffer bytes and output rows
  int64_t a_sf_bytes, b_sf_bytes, r_sf_bytes, ws_sf_bytes, y_rows;
  unsigned long long timeout_ns;
  int skip_mma;                 // test hook: the MMA warp issues nothing (waits then run out)
  unsigned long long* trace;    // nullable: stage timeline of CTA 0 (kTraceSlots per event)
};
constexpr int kTraceSlots = 64;

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Stage timeline (CTA 0 only, first kTraceSlots iterations of each event).
__device__ __forceinline__ void trace_mark(unsigned long long* trace, int event, uint32_t i) {
  if (trace && blockIdx.x == 0 && i < (uint32_t)kTraceSlots && (threadIdx.x & 31) == 0)
    trace[event * kTraceSlots + i] = global_ns();
}

// One lane of the (fully active) warp returns true.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// One 32-byte store (a whole sector) from eight 32-bit words.
__device__ __forceinline__ void st_global_32B(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand tile, rows of 128 bytes,
// 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading-dimension offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride between 8-row groups
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}
// Instruction descriptor: kind::mxf4nvf4, A and B E2M1, K-major, UE4M3 scales,
// scale-factor ids 0, dense.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// MXFP4: E8M0 scales (instruction-descriptor bit 23); each 32-bit TMEM scale
// word holds four 32-element block scales, the scale-factor id (byte 0 or 2,
// bits 29-30 for A and 4-5 for B) picks the pair a K=64 MMA uses.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, uint32_t sf_id) {
  return idesc_nvf4(M, N) | (1u << 23) | (sf_id << 29) | (sf_id << 4);
}

// The same MMA executed by the whole (converged) warp, issued by one elected lane.
__device__ __forceinline__ void tc_mma_el(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}
__device__ __forceinline__ void tc_mma_mx_el(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}
// A whole 512-element K stage (eight K = 64 MMAs over two 128-byte sub-tiles
// of A and B, 16 KB apart) issued by one elected lane in straight-line code:
// one elect for the eight MMAs (an elect per MMA costs about as much issue
// time as the MMA itself).  Descriptor start addresses advance by 32 bytes
// per K step (2 in descriptor units) and by a sub-tile (1024) after four;
// the scale columns advance by 4 per K step.
__device__ __forceinline__ void tc_mma_stage8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 a1, b1;\n\t.reg .b32 fa, fb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\tadd.u32 fa, %5, 4;\n\tadd.u32 fb, %6, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\tadd.u32 fa, %5, 8;\n\tadd.u32 fb, %6, 8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\tadd.u32 fa, %5, 12;\n\tadd.u32 fb, %6, 12;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 1024;\n\tadd.s64 b1, %2, 1024;\n\tadd.u32 fa, %5, 16;\n\tadd.u32 fb, %6, 16;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 1026;\n\tadd.s64 b1, %2, 1026;\n\tadd.u32 fa, %5, 20;\n\tadd.u32 fb, %6, 20;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 1028;\n\tadd.s64 b1, %2, 1028;\n\tadd.u32 fa, %5, 24;\n\tadd.u32 fb, %6, 24;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 1030;\n\tadd.s64 b1, %2, 1030;\n\tadd.u32 fa, %5, 28;\n\tadd.u32 fb, %6, 28;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}
__device__ __forceinline__ void tc_commit_el(uint64_t* b) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(b))
      : "memory");
}
// Descriptor of one 512-byte scale atom: 32 rows of 16 bytes, no swizzle,
// 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// Copy one scale atom into TMEM: row r of the atom (32 rows x 4 words) to lane
// r of every lane quadrant, columns taddr .. taddr+3.  Executed by the whole
// (converged) warp, issued by one elected lane.
__device__ __forceinline__ void tc_cp_sf_el(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}
// Scale atoms of two consecutive K steps (A and B) in one elected block:
// atom q to columns t, atom q+1 to t+4; B's atoms 32 columns further.  An
// atom descriptor advances by 512 bytes (32 in descriptor units) per K step.
__device__ __forceinline__ void tc_cp_sf_pair_el(uint32_t t, uint64_t da, uint64_t db) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b64 a1, b1;\n\t.reg .b32 t1, t2, t3;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "add.s64 a1, %1, 32;\n\tadd.s64 b1, %2, 32;\n\t"
      "add.u32 t1, %0, 4;\n\tadd.u32 t2, %0, 32;\n\tadd.u32 t3, %0, 36;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [t1], a1;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [t2], %2;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [t3], b1;\n\t}" ::"r"(t),
      "l"(da), "l"(db)
      : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- bounded waits
constexpr unsigned long long kDrainNs = 50000000ull;   // bound on waits for work in flight after an abort
constexpr unsigned long long kCopyDrainNs = 200000ull;  // producers' wait for their copies after an abort

struct Sync {
  volatile int* abort_flag;
  int* err;
  unsigned long long tmo;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait by one thread; `cluster` waits with cluster-scope acquire (for
// barriers another CTA arrives on).  `drain`: ignore the abort flag (used to
// let work in flight finish after an abort), still bounded by the timeout.
__device__ __forceinline__ bool wait1(uint64_t* b, uint32_t parity, const Sync& s,
                                      bool cluster = false, bool drain = false) {
  auto probe = [&]() { return cluster ? try_wait_cluster(b, parity) : mbar_try_wait(b, parity); };
  if (probe()) return true;
  const unsigned long long t0 = global_ns();
  uint32_t spins = 0;
  while (true) {
    if (probe()) return true;
    if ((++spins & 255u) == 0) {
      if (!drain && *s.abort_flag) return false;
      if (global_ns() - t0 > s.tmo) {
        if (!drain) {
          *s.abort_flag = 1;
          atomicExch(s.err, QUADS_ERR_DEVICE_TIMEOUT);
        }
        return false;
      }
    }
  }
}
// Bounded wait for a whole warp: lane 0 polls, the warp follows its verdict.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, const Sync& s,
                                          bool cluster = false) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait1(b, parity, s, cluster) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Bounded wait polled by every lane of a converged warp (the MMA warp stays
// converged for its elect-predicated tcgen05 instructions).
__device__ __forceinline__ bool conv_wait(uint64_t* b, uint32_t parity, const Sync& s,
                                          bool cluster = false) {
  auto probe = [&]() { return cluster ? try_wait_cluster(b, parity) : mbar_try_wait(b, parity); };
  if (__all_sync(0xffffffffu, probe())) return true;
  const unsigned long long t0 = global_ns();
  uint32_t spins = 0;
  while (true) {
    if (__all_sync(0xffffffffu, probe())) return true;
    if ((++spins & 255u) == 0) {
      int give_up = *s.abort_flag ? 1 : 0;
      if (!give_up && global_ns() - t0 > s.tmo) give_up = 2;
      give_up = __shfl_sync(0xffffffffu, give_up, 0);
      if (give_up) {
        if (give_up == 2 && (threadIdx.x & 31) == 0) {
          *s.abort_flag = 1;
          atomicExch(s.err, QUADS_ERR_DEVICE_TIMEOUT);
        }
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- tile schedule
struct Tile {
  int e;
  int64_t m0;   // first row of the tile in the A row space
  int n0;       // first output column
  int64_t row_end;  // rows >= row_end are not real (not stored for OUT_F32/BF16)
};

// Per-group tables copied to shared memory once per CTA (the tile decode of
// every role reads them for every tile).
struct Meta {
  int32_t* off;    // [E+1]
  int32_t* cnt;    // [E]
  float* a1;       // [E] s_a * s_w
  float* a2;       // [E] s_r * s_w
};

__device__ __forceinline__ int64_t total_tiles(const Params& p, const Meta& m) {
  if (!p.row_off) return ((p.M + BM - 1) / BM) * p.Nt;
  return (int64_t)(m.off[p.E] / BM) * p.Nt;
}

__device__ __forceinline__ Tile decode_tile(const Params& p, const Meta& m, int64_t t) {
  Tile r;
  if (!p.row_off) {
    const int64_t Mt = (p.M + BM - 1) / BM;
    r.e = 0;
    r.m0 = (t % Mt) * BM;
    r.n0 = (int)(t / Mt) * BN;
    r.row_end = p.M;
    return r;
  }
  // expert e holds tiles [off[e]/128 * Nt, off[e+1]/128 * Nt), m fastest
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)(m.off[mid] / BM) * p.Nt <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int64_t base = (int64_t)(m.off[e] / BM) * p.Nt;
  const int64_t mt_e = (m.off[e + 1] - m.off[e]) / BM;
  const int64_t local = t - base;
  r.e = e;
  r.m0 = m.off[e] + (local % mt_e) * BM;
  r.n0 = (int)(local / mt_e) * BN;
  r.row_end = m.off[e] + m.cnt[e];
  return r;
}

// ---------------------------------------------------------------- the kernel
template <class G>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmW,
                const Params p) {
  griddep_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + G::STAGES * G::STAGE_BYTES);
  uint64_t* full = bars;                           // [G::STAGES]
  uint64_t* empty = full + G::STAGES;                 // [G::STAGES]
  uint64_t* sf_ready = empty + G::STAGES;             // [G::SF_BUFS]
  uint64_t* acc_full = sf_ready + G::SF_BUFS;         // [2]
  uint64_t* acc_empty = acc_full + 2;              // [2]
  uint64_t* drain_mma = acc_empty + 2;
  uint64_t* drain_sf = drain_mma + 1;
  uint32_t* tmem_holder = (uint32_t*)(drain_sf + 1);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  Meta meta;
  meta.off = (int32_t*)(smem + G::STAGES * G::STAGE_BYTES + 1024);
  meta.cnt = meta.off + (MAX_GROUPS + 1);
  meta.a1 = (float*)(meta.cnt + MAX_GROUPS);
  meta.a2 = meta.a1 + MAX_GROUPS;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const float bts = p.mx ? 1.0f : p.b_ts[e];
    meta.a1[e] = p.mx ? 1.0f : __fmul_rn(p.a_ts[p.a_ts_pe ? e : 0], bts);
    meta.a2[e] = p.comp ? __fmul_rn(p.r_ts[p.r_ts_pe ? e : 0], bts) : 0.0f;
    if (p.row_off) {
      meta.off[e] = p.row_off[e];
      meta.cnt[e] = p.row_cnt ? p.row_cnt[e] : (p.row_off[e + 1] - p.row_off[e]);
    }
  }
  if (threadIdx.x == 0 && p.row_off) meta.off[p.E] = p.row_off[p.E];

  if (threadIdx.x == 0) {
    for (int i = 0; i < G::STAGES; ++i) { mbar_init(&full[i], G::COPIES); mbar_init(&empty[i], 1); }
    for (int i = 0; i < G::SF_BUFS; ++i) mbar_init(&sf_ready[i], SF_WARPS);
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], EPI_THREADS); }
    mbar_init(drain_mma, 1);
    mbar_init(drain_sf, SF_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const Sync sy{abort_flag, p.err, p.timeout_ns};
  const Sync dr{abort_flag, p.err, kDrainNs};

  const int64_t ntiles = total_tiles(p, meta);
  const int KT = (p.K + G::KTILE - 1) / G::KTILE;
  const int KTc = p.comp ? (p.kpad + G::KTILE - 1) / G::KTILE : 0;
  // scale bytes per 128-row block and per stage (MXFP4: one scale per 32 elements)
  const int64_t a_sf_rb = (int64_t)(p.K / (p.mx ? 128 : 64)) * 512;
  const int sf_stage = p.mx ? G::SF_TILE / 2 : G::SF_TILE;
  const int64_t r_sf_rb = (int64_t)(p.kpad / 64) * 512;

  if (warp < PRODUCERS) {
    // ------------------------------------------------------------ producers
    // A stage is ten copies: eight 8 KB code boxes (A/B x two 128-byte
    // sub-tiles x two 64-row halves) and two 4 KB scale-atom runs, dealt as
    // 3 + 3 + 4 copies so that each producer warp moves 24 KB (one warp's
    // copies are processed one after another, so the most loaded warp sets
    // the stage's pace).  Each copy arrives once on full[s] (a box with its
    // bytes, or without any when the stage's K range ends before its
    // sub-tile).  The whole warp runs the loop (so addresses and coordinates
    // stay warp-uniform); one elected lane issues.
    const int b_lo = G::copies_first(warp);
    const int b_hi = G::copies_first(warp + 1);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const Tile tl = decode_tile(p, meta, t);
      const int64_t brow = (int64_t)tl.e * p.N + tl.n0;
      for (int kt = 0; kt < KT + KTc && ok; ++kt, ++it) {
        const int s = it % G::STAGES;
        const uint32_t ph = (it / G::STAGES) & 1;
        const bool corr = kt >= KT;
        const int kk = corr ? kt - KT : kt;
        const int klen = corr ? p.kpad : p.K;
        const int ksteps = min(G::KSTEPS, (klen - kk * G::KTILE) / 64);
        const int nsub = (ksteps + 3) >> 2;   // 128-byte sub-tiles holding real columns
        uint8_t* st = smem + s * G::STAGE_BYTES;
        const CUtensorMap* ma = corr ? &tmR : &tmA;
        const CUtensorMap* mb = corr ? &tmW : &tmB;
        const uint8_t* sfa = corr ? p.r_sf + (tl.m0 / BM) * r_sf_rb : p.a_sf + (tl.m0 / BM) * a_sf_rb;
        const uint8_t* sfb = corr ? p.ws_sf + (brow / BN) * r_sf_rb : p.b_sf + (brow / BN) * a_sf_rb;
        if (!warp_wait(&empty[s], ph ^ 1, sy)) { ok = false; break; }
        if (warp == 0) trace_mark(p.trace, 0, it);
        if (elect_one()) {
          for (int b = b_lo; b < b_hi; ++b) {
            if (b >= G::BOXES) {
              const uint32_t sfbytes = (p.mx ? ksteps / 2 : ksteps) * 512;
              const uint8_t* src = (b == G::BOXES ? sfa : sfb) + kk * sf_stage;
              [[maybe_unused]] const uint8_t* base =
                  b == G::BOXES ? (corr ? p.r_sf : p.a_sf) : (corr ? p.ws_sf : p.b_sf);
              [[maybe_unused]] const int64_t lim = b == G::BOXES ? (corr ? p.r_sf_bytes : p.a_sf_bytes)
                                                              : (corr ? p.ws_sf_bytes : p.b_sf_bytes);
              if (!QDBGV(src >= base && src - base + sfbytes <= lim,
                         (tl.m0 << 20) | ((int64_t)tl.e << 8) | (corr ? 2 : 0) | (b == G::BOXES ? 0 : 4))) {
                mbar_arrive(&full[s]);   // skipped copy: the stage still completes
                continue;
              }
              mbar_expect_tx(&full[s], sfbytes);
              if (b == G::BOXES) bulk_load(st + G::A_TILE + G::B_TILE, src, sfbytes, &full[s]);
              else bulk_load(st + G::A_TILE + G::B_TILE + G::SF_TILE, src, sfbytes, &full[s]);
              continue;
            }
            const int u = b >> 2, isb = (b >> 1) & 1, hf = b & 1;
            if (u < nsub) {
              mbar_expect_tx(&full[s], BOX_BYTES);
              const int x = kk * (KSUB * G::KSUBS) + u * KSUB;
              if (isb)
                tma_load_2d(st + G::A_TILE + u * B_SUB + hf * BOX_BYTES, mb, x,
                            (int)(brow + hf * BOX_ROWS), &full[s]);
              else
                tma_load_2d(st + u * A_SUB + hf * BOX_BYTES, ma, x, (int)(tl.m0 + hf * BOX_ROWS),
                            &full[s]);
            } else {
              mbar_arrive(&full[s]);
            }
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      // the copies this warp issued land before the CTA can exit.  A stage's
      // barrier may never complete once another producer stopped before its
      // share, so the wait is a fixed bounded time (copies from L2 or HBM take
      // microseconds)
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < kCopyDrainNs) {
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_nvf4(BM, BN);
    uint32_t s = 0, sb = 0, sph = 0;
    uint32_t j = 0, mit = 0;
    bool ok = !p.skip_mma;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++j) {
      const uint32_t b = j & 1;
      if (!conv_wait(&acc_empty[b], ((j >> 1) & 1) ^ 1, sy)) { ok = false; break; }
      tc_fence_after();
      for (int kt = 0; kt < KT + KTc; ++kt) {
        const bool corr = kt >= KT;
        const int kk = corr ? kt - KT : kt;
        if (corr && kk == 0 && j > 0) {
          // acc2 is free once the previous tile's epilogue is done
          if (!conv_wait(&acc_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, sy)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // the staging warps saw this stage's TMA data land (full[s]) and have
        // written its scales into TMEM buffer sb: one barrier covers both
        if (!conv_wait(&sf_ready[sb], sph, sy)) { ok = false; break; }
        trace_mark(p.trace, 3, mit);
        tc_fence_after();
        const int klen = corr ? p.kpad : p.K;
        const int ksteps = min(G::KSTEPS, (klen - kk * G::KTILE) / 64);
        const uint32_t sa = smem_u32(smem + s * G::STAGE_BYTES);
        const uint32_t sbb = sa + G::A_TILE;
        const uint32_t tsf = tmem + SF_COL + sb * G::SF_BUF_COLS;
        const uint32_t dcol = corr ? (tmem + ACC2_COL) : (tmem + b * BN);
        if (p.mx) {
          for (int q = 0; q < ksteps; ++q) {
            const uint32_t off = (q >> 2) * A_SUB + (q & 3) * 32;
            const uint32_t id = (q & 1) ? idesc_mxf4(BM, BN, 2) : idesc_mxf4(BM, BN, 0);
            tc_mma_mx_el(dcol, desc_sw128(sa + off), desc_sw128(sbb + off), id,
                         tsf + (q >> 1) * 4, tsf + 4 * G::KSTEPS + (q >> 1) * 4,
                         (kk > 0 || q > 0) ? 1u : 0u);
          }
        } else if (G::KSTEPS == 8 && ksteps == 8) {
          tc_mma_stage8(dcol, desc_sw128(sa), desc_sw128(sbb), idesc, tsf, tsf + 4 * G::KSTEPS,
                        kk > 0 ? 1u : 0u);
        } else {
          for (int q = 0; q < ksteps; ++q) {
            const uint32_t off = (q >> 2) * A_SUB + (q & 3) * 32;
            tc_mma_el(dcol, desc_sw128(sa + off), desc_sw128(sbb + off), idesc, tsf + q * 4,
                      tsf + 4 * G::KSTEPS + q * 4, (kk > 0 || q > 0) ? 1u : 0u);
          }
        }
        tc_commit_el(&empty[s]);   // also frees this stage's scale buffer
        trace_mark(p.trace, 4, mit++);
        if (++s == G::STAGES) s = 0;
        if (++sb == G::SF_BUFS) { sb = 0; sph ^= 1; }
      }
      if (!ok) break;
      tc_commit_el(&acc_full[b]);
    }
    // every MMA this warp issued completes before TMEM or shared memory go away
    tc_commit_el(drain_mma);
    if (lane == 0) wait1(drain_mma, 0, dr, false, true);
    __syncwarp();
  } else if (warp >= SF_WARP0 && warp < EPI_WARP0) {
    // ------------------------------------------------------------ scale staging
    // TMEM buffer sb holds, at column SF_COL + 64*sb + 4*q + j (A) and +32 (B),
    // lane l of every quadrant, the scale word of row l + 32*j for K step q --
    // row l of scale atom q -- the layout the block-scaled MMA reads (row r's
    // four scales at lane r % 32, column r / 32).  Warp w copies the atoms of
    // K steps 2w and 2w+1.  The warps wait for the stage's TMA data, so
    // sf_ready alone tells the MMA warp that the stage is complete.
    // Scale buffer sb was last read by the MMAs of ring iteration it - G::SF_BUFS,
    // whose completion the MMA warp signals on that stage's empty barrier.
    const int w = warp - SF_WARP0;
    uint32_t s = 0, ph = 0, sb = 0, it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      for (int kt = 0; kt < KT + KTc; ++kt, ++it) {
        bool okw = conv_wait(&full[s], ph, sy);
        if (okw && it >= (uint32_t)G::SF_BUFS) {
          const uint32_t prev = it - G::SF_BUFS;
          okw = conv_wait(&empty[prev % G::STAGES], (prev / G::STAGES) & 1, sy);
        }
        if (!okw) {
          ok = false;
          break;
        }
        if (w == 0) trace_mark(p.trace, 1, it);
        tc_fence_after();
        const bool corr = kt >= KT;
        const int kk = corr ? kt - KT : kt;
        const int klen = corr ? p.kpad : p.K;
        const int ksteps = min(G::KSTEPS, (klen - kk * G::KTILE) / 64);
        const uint32_t ssf = smem_u32(smem + s * G::STAGE_BYTES + G::A_TILE + G::B_TILE);
        const uint32_t tsf = tmem + SF_COL + sb * G::SF_BUF_COLS;
        if (p.mx) {
          // MXFP4: one atom covers two K steps; warp w copies atom w
          if (2 * w < ksteps) {
            tc_cp_sf_el(tsf + w * 4, desc_sf(ssf + w * 512));
            tc_cp_sf_el(tsf + 4 * G::KSTEPS + w * 4, desc_sf(ssf + G::SF_TILE + w * 512));
          }
        } else if (G::KSTEPS == 2 * SF_WARPS && 4 * G::KSTEPS == 32 && 2 * w + 1 < ksteps) {
          const int q = 2 * w;
          tc_cp_sf_pair_el(tsf + q * 4, desc_sf(ssf + q * 512), desc_sf(ssf + G::SF_TILE + q * 512));
        } else {
#pragma unroll
          for (int i = 0; i < G::KSTEPS / SF_WARPS; ++i) {
            const int q = w * (G::KSTEPS / SF_WARPS) + i;
            if (q < ksteps) {
              tc_cp_sf_el(tsf + q * 4, desc_sf(ssf + q * 512));
              tc_cp_sf_el(tsf + 4 * G::KSTEPS + q * 4, desc_sf(ssf + G::SF_TILE + q * 512));
            }
          }
        }
        tc_commit_el(&sf_ready[sb]);
        if (w == 0) trace_mark(p.trace, 2, it);
        if (++s == G::STAGES) { s = 0; ph ^= 1; }
        if (++sb == G::SF_BUFS) sb = 0;
      }
    }
    // the scale copies this warp issued complete before TMEM goes away
    tc_commit_el(drain_sf);
    if (lane == 0) wait1(drain_sf, 0, dr, false, true);
    __syncwarp();
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
    const int half = (warp - EPI_WARP0) >> 2;  // which half of the tile's columns
    const int row_in_tile = quad * 32 + lane;
    uint32_t j = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
      const Tile tl = decode_tile(p, meta, t);
      const uint32_t b = j & 1;
      // lane 0 waits, the warp follows it (tcgen05.ld needs the whole warp)
      if (!warp_wait(&acc_full[b], (j >> 1) & 1, sy)) break;
      if (warp == EPI_WARP0) trace_mark(p.trace, 5, j);
      tc_fence_after();
      const float a1 = meta.a1[tl.e];
      const float a2 = meta.a2[tl.e];
      const int64_t row = tl.m0 + row_in_tile;
      const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
      const uint32_t t1 = tmem + lane_base + b * BN;
      const uint32_t t2 = tmem + lane_base + ACC2_COL;
      float amax = 0.0f;
      if (p.out_mode == OUT_SWIGLU) {
        // tile columns [0,64) are gate rows of W, [64,128) the matching up rows;
        // this warp produces h columns [32*half, 32*half + 32) of the tile
        const bool store = row < (p.row_off ? (int64_t)meta.off[tl.e + 1] : p.M) && QDBG(row < p.y_rows);
        __nv_bfloat16* y = (__nv_bfloat16*)p.y + row * p.ldy + tl.n0 / 2;
#pragma unroll 1
        for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
          float g1[16], u1[16], g2[16], u2[16];
          __syncwarp();  // tcgen05.ld is warp-collective: the row-masked stores above diverge
          tc_ld16(t1 + c0, g1);
          tc_ld16(t1 + 64 + c0, u1);
          if (p.comp) { tc_ld16(t2 + c0, g2); tc_ld16(t2 + 64 + c0, u2); }
          tc_wait_ld();
          if (c0 + 16 == half * 32 + 32) {
            // the last TMEM read of this tile is done: release the accumulators
            // before the math and the stores, so the next MMAs can start
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
          }
          uint32_t packed[8];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float h[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              float g = a1 * g1[i + q], u = a1 * u1[i + q];
              if (p.comp) { g = fmaf(a2, g2[i + q], g); u = fmaf(a2, u2[i + q], u); }
              h[q] = __fdividef(g * u, 1.0f + __expf(-g));   // silu(g) * u
            }
            __nv_bfloat162 hb = __floats2bfloat162_rn(h[0], h[1]);
            packed[i / 2] = *reinterpret_cast<uint32_t*>(&hb);
            const float2 hr = __bfloat1622float2(hb);
            amax = fmaxf(amax, fmaxf(fabsf(hr.x), fabsf(hr.y)));
          }
          if (store) {
            if (p.st32) {
              st_global_32B(y + c0, packed);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(y + c0);
              dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
              dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
          }
        }
        if (!store) amax = 0.0f;
      } else {
        const bool store = row < tl.row_end && QDBG(row < p.y_rows);
#pragma unroll 1
        for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
          float v1[16], v2[16];
          __syncwarp();  // tcgen05.ld is warp-collective: the row-masked stores above diverge
          tc_ld16(t1 + c0, v1);
          if (p.comp) tc_ld16(t2 + c0, v2);
          tc_wait_ld();
          if (c0 + 16 == half * 64 + 64) {
            // the last TMEM read of this tile is done: release the accumulators
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
          }
          float o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = p.comp ? fmaf(a2, v2[i], a1 * v1[i]) : a1 * v1[i];
          if (store) {
            if (p.out_mode == OUT_F32) {
              float* yrow = (float*)p.y + row * p.ldy + tl.n0 + c0;
              if (p.st32) {
                st_global_32B(yrow, reinterpret_cast<const uint32_t*>(o));
                st_global_32B(yrow + 8, reinterpret_cast<const uint32_t*>(o + 8));
              } else {
                float4* dst = reinterpret_cast<float4*>(yrow);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(o[i]));
            } else {
              uint32_t packed[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                __nv_bfloat162 hb = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
                packed[i] = *reinterpret_cast<uint32_t*>(&hb);
                const float2 hr = __bfloat1622float2(hb);
                amax = fmaxf(amax, fmaxf(fabsf(hr.x), fabsf(hr.y)));
              }
              __nv_bfloat16* yrow = (__nv_bfloat16*)p.y + row * p.ldy + tl.n0 + c0;
              if (p.st32) {
                st_global_32B(yrow, packed);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(yrow);
                dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (warp == EPI_WARP0) trace_mark(p.trace, 6, j);
      if (p.y_amax) {
        amax = warp_max(amax);
        if (lane == 0 && amax > 0.0f) atomicMax(&p.y_amax[tl.e], __float_as_uint(amax));
      }
    }
  }
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
  }
}

// ---------------------------------------------------------------- CTA-pair kernel
// The same product on pairs of SMs: a 2-CTA cluster issues
// tcgen05.mma.cta_group::2 with M = 256 (each CTA holds 128 rows of A and
// the accumulator rows of its half) and N = 128 (each CTA holds 64 of the
// 128 rows of B; the tensor cores read both halves).  Per SM that is the
// work of a 128 x 128 tile for 3/4 of the operand bytes, so each 512-element
// K stage is 56 KB and four stages fit where three did.
//
// A tile's K stream is a sequence of 256-element sub-tiles -- the main K
// range, then the k-channel correction -- packed two per ring stage, so the
// correction shares a stage with the main loop's last sub-tile when there is
// room (K = 768: two stages per tile instead of three).
//
// Roles (16 warps per CTA):
//   warps 0-3  TMA producers of this CTA's operands (A rows, its 64 rows of
//              B, the scale atoms).  Every copy of both CTAs completes on the
//              leader's full barrier of the stage (cp.async.bulk.tensor
//              .cta_group::2 names the leader's barrier); the leader's first
//              producer expects the bytes of both CTAs, so no CTA has to
//              forward anything to the other.
//   warp 4     TMEM allocation (both CTAs); leader: the MMA issuer.
//   warps 5-6  leader: scale atoms of a stage into TMEM of both CTAs
//              (tcgen05.cp.cta_group::2), one sub-tile each.
//   warps 8-15 epilogue of this CTA's 128 rows (two warps per lane quadrant).
// The leader's MMA commits free a stage in both CTAs and announce a full
// accumulator to both; both CTAs' epilogues arrive on the leader's
// accumulator-empty barrier.  Every wait is bounded; on a timeout a CTA stops
// its roles, lets its copies and tensor-core work in flight finish (the
// leader waits for them on its barriers, with a bound; the peer, whose copies
// complete on the leader's barriers, waits a fixed bounded time), meets its
// peer at the cluster barrier and frees its TMEM.
namespace pair {

constexpr int BM = 128;                       // rows of A per CTA (M = 256 per pair)
constexpr int BN = 128;                       // output columns of a pair tile
constexpr int BNH = 64;                       // rows of B held by each CTA
constexpr int KSUB = 128;                     // bytes per row of a 128B-swizzled sub-tile (256 FP4)
constexpr int SLOTS = 2;                      // sub-tiles per stage
constexpr int STAGES = 4;
constexpr int A_SUB = BM * KSUB;              // 16 KB
constexpr int B_SUB = BNH * KSUB;             // 8 KB
constexpr int SF_SUB = 4 * 512;               // four 128-row scale atoms (one per K = 64 step)
constexpr int OFF_B = SLOTS * A_SUB;
constexpr int OFF_SFA = OFF_B + SLOTS * B_SUB;
constexpr int OFF_SFB = OFF_SFA + SLOTS * SF_SUB;
constexpr int STAGE_BYTES = OFF_SFB + SLOTS * SF_SUB;   // 56 KB
constexpr int BOX_ROWS = 64;
constexpr int BOX_BYTES = BOX_ROWS * KSUB;    // 8 KB
constexpr int PRODUCERS = 4;
constexpr int SF_BOX_ROWS = SF_SUB / 128;     // a sub-tile's atoms as 128-byte rows (TMA box)
constexpr int MMA_WARP = 4, SF_WARP0 = 5, SF_WARPS = 2, EPI_WARP0 = 8;
constexpr int NUM_THREADS = 512;
constexpr int EPI_WARPS = 8;
constexpr int TMEM_COLS = 512;
constexpr int ACC2_COL = 256;
constexpr int SF_COL = 384;
constexpr int SF_BUFS = 2;
constexpr int SF_BUF_COLS = 64;               // A atoms at +4a, B atoms at +32+4a (a < 8)
constexpr int MAX_GROUPS = 256;
constexpr int NBARS = 2 * STAGES + SF_BUFS + 4 + 2;
constexpr int BAR_BYTES = NBARS * 8 + 16;     // + TMEM holder and abort flag
constexpr int META_BYTES = 4 * (MAX_GROUPS + 1);
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + META_BYTES + 1024 /*align*/;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

struct Params {
  int E, N, K, kpad, Nt;
  int64_t M;                    // dense rows (row_off == nullptr)
  const int32_t* row_off;       // [E+1] padded row offsets (multiples of 128) or null
  const int32_t* row_cnt;       // [E] real rows (null: whole groups)
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const uint8_t* r_sf;
  const uint8_t* ws_sf;
  const float* a_ts;
  const float* b_ts;
  const float* r_ts;
  int a_ts_pe, r_ts_pe;
  int comp;
  int mx;
  void* y;
  int64_t ldy;
  int out_mode;
  int st32;
  uint32_t* y_amax;
  int* err;
  unsigned long long timeout_ns;
  int skip_mma;                 // test hook: the MMA warp issues nothing (waits then run out)
  // extents for the bounds-checked build: scale buffer bytes and output rows
  int64_t a_sf_bytes, b_sf_bytes, r_sf_bytes, ws_sf_bytes, y_rows;
  unsigned long long* trace;    // nullable: stage timeline of the first pair's leader
};

__device__ __forceinline__ void mma_nvf4_cg2(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}
__device__ __forceinline__ void mma_mxf4_cg2(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}
// The four K = 64 MMAs of one 256-element sub-tile under one elect (see
// tc_mma_stage8): descriptors +2 per K step, scale columns +4.
__device__ __forceinline__ void mma_nvf4_cg2_x4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 a1, b1;\n\t.reg .b32 fa, fb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\tadd.u32 fa, %5, 4;\n\tadd.u32 fb, %6, 4;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\tadd.u32 fa, %5, 8;\n\tadd.u32 fb, %6, 8;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\tadd.u32 fa, %5, 12;\n\tadd.u32 fb, %6, 12;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}
// Four scale atoms of A (columns ta + 4a) and four of B (tb + 4a), atom
// descriptors +32 per atom, under one elect.
__device__ __forceinline__ void cp_sf_cg2_x4(uint32_t ta, uint32_t tb, uint64_t da, uint64_t db) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b64 x;\n\t.reg .b32 t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %2;\n\t"
      "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%1], %3;\n\t"
      "add.s64 x, %2, 32;\n\tadd.u32 t, %0, 4;\n\t@e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], x;\n\t"
      "add.s64 x, %3, 32;\n\tadd.u32 t, %1, 4;\n\t@e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], x;\n\t"
      "add.s64 x, %2, 64;\n\tadd.u32 t, %0, 8;\n\t@e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], x;\n\t"
      "add.s64 x, %3, 64;\n\tadd.u32 t, %1, 8;\n\t@e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], x;\n\t"
      "add.s64 x, %2, 96;\n\tadd.u32 t, %0, 12;\n\t@e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], x;\n\t"
      "add.s64 x, %3, 96;\n\tadd.u32 t, %1, 12;\n\t@e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], x;\n\t}"
      ::"r"(ta), "r"(tb), "l"(da), "l"(db)
      : "memory");
}
// Commit of the executing thread's earlier tcgen05 work: arrive on the
// barrier at the same offset in every CTA of `mask`.
__device__ __forceinline__ void commit_mc_cg2(uint64_t* b, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(smem_u32(b)),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void cp_sf_cg2(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}

// TMA load into this CTA's shared memory that completes on the barrier at
// cluster address `bar` (the leader's).
__device__ __forceinline__ void tma_load_2d_cg2(void* dst, const CUtensorMap* map, int x, int y,
                                                uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// A pair tile: rows [m0, m0 + 256) (the peer's half starts at m0 + 128) x
// output columns [n0, n0 + 128) of group e.
struct Tile {
  int e;
  int64_t m0;
  int n0;
  int64_t row_end;   // rows >= row_end are not stored (plain / f32 outputs)
  int64_t grp_end;   // end of the group's padded rows (SwiGLU stores up to here)
  int64_t blk_lim;   // 128-row blocks >= blk_lim hold none of the group's rows
};

__device__ __forceinline__ int64_t total_tiles(const Params& p, const int32_t* poff) {
  if (!p.row_off) return ((p.M + 2 * BM - 1) / (2 * BM)) * p.Nt;
  return (int64_t)poff[p.E] * p.Nt;
}

__device__ __forceinline__ Tile decode_tile(const Params& p, const int32_t* poff, int64_t t) {
  Tile r;
  if (!p.row_off) {
    const int64_t Mt = (p.M + 2 * BM - 1) / (2 * BM);
    r.e = 0;
    r.m0 = (t % Mt) * 2 * BM;
    r.n0 = (int)(t / Mt) * BN;
    r.row_end = p.M;
    r.grp_end = p.M;
    r.blk_lim = (p.M + BM - 1) / BM;
    return r;
  }
  // group e holds pair tiles [poff[e] * Nt, poff[e+1] * Nt), m fastest
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)poff[mid] * p.Nt <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int64_t pairs = poff[e + 1] - poff[e];
  const int64_t local = t - (int64_t)poff[e] * p.Nt;
  const int64_t o0 = __ldg(p.row_off + e), o1 = __ldg(p.row_off + e + 1);
  (void)QDBGV(o0 >= 0 && o0 <= o1 && o1 <= p.y_rows && pairs > 0, (o1 << 16) | e);
  r.e = e;
  r.m0 = o0 + (local % pairs) * 2 * BM;
  r.n0 = (int)(local / pairs) * BN;
  r.row_end = o0 + (p.row_cnt ? __ldg(p.row_cnt + e) : (o1 - o0));
  r.grp_end = o1;
  r.blk_lim = o1 / BM;
  return r;
}

// Sub-tile j of a tile's K stream: main K sub-tiles first, then the
// correction's.  Returns the number of K = 64 steps it holds (0: empty slot).
struct Sub {
  int ksteps;
  bool corr;
  int kk;        // sub-tile index inside its own K range
};
__device__ __forceinline__ Sub sub_of(const Params& p, int j, int nmain, int ncorr) {
  Sub s;
  if (j < nmain) {
    s.corr = false;
    s.kk = j;
    s.ksteps = min(4, (p.K - j * 256) / 64);
  } else if (j < nmain + ncorr) {
    s.corr = true;
    s.kk = j - nmain;
    s.ksteps = min(4, (p.kpad - s.kk * 256) / 64);
  } else {
    s.corr = false;
    s.kk = 0;
    s.ksteps = 0;
  }
  return s;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmR,
                     const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tsA,
                     const __grid_constant__ CUtensorMap tsB,
                     const __grid_constant__ CUtensorMap tsR,
                     const __grid_constant__ CUtensorMap tsW, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;                                 // [STAGES] (leader's: both CTAs' copies)
  uint64_t* empty = full + STAGES;                       // [STAGES]
  uint64_t* sf_ready = empty + STAGES;                   // [SF_BUFS] (leader)
  uint64_t* acc_full = sf_ready + SF_BUFS;               // [2]
  uint64_t* acc_empty = acc_full + 2;                    // [2] (leader)
  uint64_t* drain_mma = acc_empty + 2;                   // leader
  uint64_t* drain_sf = drain_mma + 1;                    // leader
  uint32_t* tmem_holder = (uint32_t*)(drain_sf + 1);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  int32_t* poff = (int32_t*)(smem + STAGES * STAGE_BYTES + BAR_BYTES);   // [E+1] pair prefix

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const Sync sy{abort_flag, p.err, p.timeout_ns};

  // pair prefix of the groups: pairs_e = ceil(blocks_e / 2), exclusive scan
  if (p.row_off && warp < 8) {
    __shared__ int wsum[8];
    const int e = threadIdx.x;   // warps 0-7 cover up to 256 groups
    int v = 0;
    if (e < p.E) {
      const int blocks = (__ldg(p.row_off + e + 1) - __ldg(p.row_off + e)) / BM;
      v = (blocks + 1) >> 1;
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    int before = 0;
    for (int i = 0; i < warp; ++i) before += wsum[i];
    if (e < p.E) poff[e + 1] = before + incl;
    if (e == 0) poff[0] = 0;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // the leader's expect_tx; the copies complete the bytes
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < SF_BUFS; ++i) mbar_init(&sf_ready[i], SF_WARPS);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 2 * EPI_WARPS);
    }
    mbar_init(drain_mma, 1);
    mbar_init(drain_sf, SF_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    // one warp of each CTA of the pair allocates, collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int64_t ntiles = total_tiles(p, poff);
  const int64_t cid = cluster_id(), ncl = cluster_count();
  const int nmain = (p.K + 255) / 256;
  const int ncorr = p.comp ? (p.kpad + 255) / 256 : 0;
  const int nst = (nmain + ncorr + SLOTS - 1) / SLOTS;   // ring stages per tile
  // scale bytes per 128-row block and per 256-element sub-tile
  const int64_t a_sf_rb = (int64_t)(p.K / (p.mx ? 128 : 64)) * 512;
  const int64_t r_sf_rb = (int64_t)(p.kpad / 64) * 512;
  const int sf_sub = p.mx ? SF_SUB / 2 : SF_SUB;

  if (warp < PRODUCERS) {
    // ---------------------------------------------------------- producers
    // warp 0: A boxes of slot 0, warp 1: A boxes of slot 1, warp 2: the B box
    // of both slots, warp 3: the scale atoms (A and B) of both slots.  The
    // leader's warp 0 expects the stage's bytes of both CTAs before its own
    // copies; the other copies may land first (the barrier's transaction
    // count then runs ahead, which it allows).
    const uint32_t full0 = peer_addr(&full[0], 0);
    const uint32_t sf_box = (p.mx ? SF_BOX_ROWS / 2 : SF_BOX_ROWS) * 128;
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = cid; t < ntiles && ok; t += ncl) {
      const Tile tl = decode_tile(p, poff, t);
      const int64_t mrow = tl.m0 + (int64_t)rank * BM;          // this CTA's A rows
      int64_t blk = mrow / BM;                                  // its scale rows
      if (blk >= tl.blk_lim) blk = tl.m0 / BM;                  // no rows of the group: any valid block
      const int64_t bbase = (int64_t)tl.e * p.N + tl.n0;        // the pair's 128 B rows
      const int64_t brow = bbase + (int64_t)rank * BNH;         // this CTA's 64 of them
      for (int kt = 0; kt < nst && ok; ++kt, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!warp_wait(&empty[s], ph ^ 1, sy)) { ok = false; break; }
        if (warp == 0) trace_mark(p.trace, 0, it);
        uint8_t* st = smem + s * STAGE_BYTES;
        const uint32_t bar = full0 + 8u * s;
        if (elect_one()) {
          if (leader && warp == 0) {
            uint32_t bytes = 0;
            for (int u = 0; u < SLOTS; ++u)
              if (sub_of(p, kt * SLOTS + u, nmain, ncorr).ksteps)
                bytes += A_SUB + B_SUB + 2 * sf_box;
            mbar_expect_tx(&full[s], 2 * bytes);   // both CTAs
          }
          for (int u = 0; u < SLOTS; ++u) {
            const Sub sb = sub_of(p, kt * SLOTS + u, nmain, ncorr);
            if (!sb.ksteps) continue;
            const CUtensorMap* ma = sb.corr ? &tmR : &tmA;
            const CUtensorMap* mb = sb.corr ? &tmW : &tmB;
            const int x = sb.kk * KSUB;
            if (warp == u) {            // A: two 64-row boxes
              for (int h = 0; h < 2; ++h)
                tma_load_2d_cg2(st + u * A_SUB + h * BOX_BYTES, ma, x, (int)(mrow + h * BOX_ROWS), bar);
            } else if (warp == 2) {     // B: this CTA's 64 rows
              tma_load_2d_cg2(st + OFF_B + u * B_SUB, mb, x, (int)brow, bar);
            } else if (warp == 3) {     // scale atoms of A and of the pair's B, as 128-byte rows
              const int64_t oa = sb.corr ? blk * r_sf_rb + (int64_t)sb.kk * SF_SUB
                                         : blk * a_sf_rb + (int64_t)sb.kk * sf_sub;
              const int64_t ow = sb.corr ? (bbase / BM) * r_sf_rb + (int64_t)sb.kk * SF_SUB
                                         : (bbase / BM) * a_sf_rb + (int64_t)sb.kk * sf_sub;
              (void)QDBGV(oa >= 0 && oa + sf_box <= (sb.corr ? p.r_sf_bytes : p.a_sf_bytes) + 3 * 512,
                          (tl.m0 << 20) | ((int64_t)tl.e << 8) | (sb.corr ? 2 : 0) | (int)rank);
              (void)QDBGV(ow >= 0 && ow + sf_box <= (sb.corr ? p.ws_sf_bytes : p.b_sf_bytes) + 3 * 512,
                          (bbase << 20) | ((int64_t)tl.e << 8) | (sb.corr ? 2 : 0) | 4 | (int)rank);
              tma_load_2d_cg2(st + OFF_SFA + u * SF_SUB, sb.corr ? &tsR : &tsA, 0, (int)(oa / 128), bar);
              tma_load_2d_cg2(st + OFF_SFB + u * SF_SUB, sb.corr ? &tsW : &tsB, 0, (int)(ow / 128), bar);
            }
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      // let the copies this CTA issued land before it can exit: the leader
      // waits for the stages' barriers (bounded); the peer, whose copies
      // complete on the leader's barriers, waits a fixed bounded time
      if (leader) {
        const Sync dr{abort_flag, p.err, kDrainNs};
        const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j) wait1(&full[j % STAGES], (j / STAGES) & 1, dr, false, true);
      } else {
        const unsigned long long t0 = global_ns();
        while (global_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == MMA_WARP && leader) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_nvf4(2 * BM, BN);
    uint32_t s = 0, sb = 0, sph = 0, j = 0, mit = 0;
    bool ok = !p.skip_mma;
    for (int64_t t = cid; t < ntiles && ok; t += ncl, ++j) {
      const uint32_t b = j & 1;
      if (!conv_wait(&acc_empty[b], ((j >> 1) & 1) ^ 1, sy, true)) { ok = false; break; }
      tc_fence_after();
      for (int kt = 0; kt < nst; ++kt) {
        if (!conv_wait(&sf_ready[sb], sph, sy)) { ok = false; break; }
        trace_mark(p.trace, 3, mit);
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
        const uint32_t tsf = tmem + SF_COL + sb * SF_BUF_COLS;
        for (int u = 0; u < SLOTS; ++u) {
          const int jj = kt * SLOTS + u;
          const Sub sub = sub_of(p, jj, nmain, ncorr);
          if (!sub.ksteps) continue;
          if (sub.corr && sub.kk == 0 && j > 0) {
            // acc2 is free once the previous tile's epilogues are done
            if (!conv_wait(&acc_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, sy, true)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t dcol = sub.corr ? (tmem + ACC2_COL) : (tmem + b * BN);
          const bool first_sub = sub.corr ? (sub.kk == 0) : (jj == 0);
          const uint32_t a0 = sa + u * A_SUB, b0 = sa + OFF_B + u * B_SUB;
          if (!p.mx && sub.ksteps == 4) {
            mma_nvf4_cg2_x4(dcol, desc_sw128(a0), desc_sw128(b0), idesc, tsf + 16 * u,
                            tsf + 32 + 16 * u, first_sub ? 0u : 1u);
            continue;
          }
          for (int q = 0; q < sub.ksteps; ++q) {
            const uint32_t acc = (first_sub && q == 0) ? 0u : 1u;
            if (p.mx) {
              const uint32_t at = 2 * u + (q >> 1);
              const uint32_t id = (q & 1) ? idesc_mxf4(2 * BM, BN, 2) : idesc_mxf4(2 * BM, BN, 0);
              mma_mxf4_cg2(dcol, desc_sw128(a0 + q * 32), desc_sw128(b0 + q * 32), id,
                           tsf + 4 * at, tsf + 32 + 4 * at, acc);
            } else {
              const uint32_t at = 4 * u + q;
              mma_nvf4_cg2(dcol, desc_sw128(a0 + q * 32), desc_sw128(b0 + q * 32), idesc,
                           tsf + 4 * at, tsf + 32 + 4 * at, acc);
            }
          }
        }
        if (!ok) break;
        commit_mc_cg2(&empty[s], 0x3);   // frees the stage in both CTAs (and the scale buffer)
        trace_mark(p.trace, 4, mit++);
        if (++s == STAGES) s = 0;
        if (++sb == SF_BUFS) { sb = 0; sph ^= 1; }
      }
      if (!ok) break;
      commit_mc_cg2(&acc_full[b], 0x3);
    }
    // every MMA this thread issued has completed before TMEM or shared memory go away
    commit_mc_cg2(drain_mma, 0x1);
    if (lane == 0) wait1(drain_mma, 0, Sync{abort_flag, p.err, kDrainNs}, false, true);
    __syncwarp();
  } else if (warp >= SF_WARP0 && warp < SF_WARP0 + SF_WARPS && leader) {
    // ---------------------------------------------------------- scale staging
    // Warp w copies slot w's scale atoms of a stage once both CTAs' copies
    // have landed; scale buffer sb was last read by the MMAs of ring
    // iteration it - SF_BUFS (signalled on that stage's empty barrier).
    const int w = warp - SF_WARP0;
    uint32_t s = 0, ph = 0, sb = 0, it = 0;
    bool ok = true;
    for (int64_t t = cid; t < ntiles && ok; t += ncl) {
      for (int kt = 0; kt < nst; ++kt, ++it) {
        bool okw = conv_wait(&full[s], ph, sy, true);
        if (okw && it >= (uint32_t)SF_BUFS) {
          const uint32_t prev = it - SF_BUFS;
          okw = conv_wait(&empty[prev % STAGES], (prev / STAGES) & 1, sy);
        }
        if (!okw) { ok = false; break; }
        if (w == 0) trace_mark(p.trace, 1, it);
        tc_fence_after();
        const Sub sub = sub_of(p, kt * SLOTS + w, nmain, ncorr);
        const uint32_t ssa = smem_u32(smem + s * STAGE_BYTES + OFF_SFA + w * SF_SUB);
        const uint32_t ssb = smem_u32(smem + s * STAGE_BYTES + OFF_SFB + w * SF_SUB);
        const uint32_t tsf = tmem + SF_COL + sb * SF_BUF_COLS;
        const int natoms = p.mx ? (sub.ksteps + 1) / 2 : sub.ksteps;
        const int abase = p.mx ? 2 * w : 4 * w;
        if (natoms == 4) {
          cp_sf_cg2_x4(tsf + 4 * abase, tsf + 32 + 4 * abase, desc_sf(ssa), desc_sf(ssb));
        } else
        for (int a = 0; a < natoms; ++a) {
          cp_sf_cg2(tsf + 4 * (abase + a), desc_sf(ssa + a * 512));
          cp_sf_cg2(tsf + 32 + 4 * (abase + a), desc_sf(ssb + a * 512));
        }
        commit_mc_cg2(&sf_ready[sb], 0x1);
        if (w == 0) trace_mark(p.trace, 2, it);
        if (++s == STAGES) { s = 0; ph ^= 1; }
        if (++sb == SF_BUFS) sb = 0;
      }
    }
    commit_mc_cg2(drain_sf, 0x1);
    if (lane == 0) wait1(drain_sf, 0, Sync{abort_flag, p.err, kDrainNs}, false, true);
    __syncwarp();
  } else if (warp >= EPI_WARP0) {
    // ---------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int half = (warp - EPI_WARP0) >> 2;
    const int row_in_tile = (int)rank * BM + quad * 32 + lane;
    const uint32_t acc_empty_leader = peer_addr(&acc_empty[0], 0);
    uint32_t j = 0;
    for (int64_t t = cid; t < ntiles; t += ncl, ++j) {
      const Tile tl = decode_tile(p, poff, t);
      const uint32_t b = j & 1;
      if (!warp_wait(&acc_full[b], (j >> 1) & 1, sy, true)) break;
      if (warp == EPI_WARP0) trace_mark(p.trace, 5, j);
      tc_fence_after();
      const float bts = p.mx ? 1.0f : __ldg(p.b_ts + tl.e);
      const float a1 = p.mx ? 1.0f : __fmul_rn(__ldg(p.a_ts + (p.a_ts_pe ? tl.e : 0)), bts);
      const float a2 = p.comp ? __fmul_rn(__ldg(p.r_ts + (p.r_ts_pe ? tl.e : 0)), bts) : 0.0f;
      const int64_t row = tl.m0 + row_in_tile;
      const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
      const uint32_t t1 = tmem + lane_base + b * BN;
      const uint32_t t2 = tmem + lane_base + ACC2_COL;
      auto release = [&]() {
        // this warp's last TMEM read of the tile is done: tell the leader
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&acc_empty[b]);
          else arrive_cluster(acc_empty_leader + 8u * b);
        }
      };
      float amax = 0.0f;
      if (p.out_mode == OUT_SWIGLU) {
        // tile columns [0,64) are gate rows of W, [64,128) the matching up rows;
        // this warp produces h columns [32*half, 32*half + 32) of the tile
        const bool store = row < tl.grp_end && QDBG(row < p.y_rows);
        __nv_bfloat16* y = (__nv_bfloat16*)p.y + row * p.ldy + tl.n0 / 2;
#pragma unroll 1
        for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
          float g1[16], u1[16], g2[16], u2[16];
          __syncwarp();
          tc_ld16(t1 + c0, g1);
          tc_ld16(t1 + 64 + c0, u1);
          if (p.comp) { tc_ld16(t2 + c0, g2); tc_ld16(t2 + 64 + c0, u2); }
          tc_wait_ld();
          if (c0 + 16 == half * 32 + 32) release();
          uint32_t packed[8];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float h[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              float g = a1 * g1[i + q], u = a1 * u1[i + q];
              if (p.comp) { g = fmaf(a2, g2[i + q], g); u = fmaf(a2, u2[i + q], u); }
              h[q] = __fdividef(g * u, 1.0f + __expf(-g));   // silu(g) * u
            }
            __nv_bfloat162 hb = __floats2bfloat162_rn(h[0], h[1]);
            packed[i / 2] = *reinterpret_cast<uint32_t*>(&hb);
            const float2 hr = __bfloat1622float2(hb);
            amax = fmaxf(amax, fmaxf(fabsf(hr.x), fabsf(hr.y)));
          }
          if (store) {
            if (p.st32) {
              st_global_32B(y + c0, packed);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(y + c0);
              dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
              dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
          }
        }
        if (!store) amax = 0.0f;
      } else {
        const bool store = row < tl.row_end && QDBG(row < p.y_rows);
#pragma unroll 1
        for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
          float v1[16], v2[16];
          __syncwarp();
          tc_ld16(t1 + c0, v1);
          if (p.comp) tc_ld16(t2 + c0, v2);
          tc_wait_ld();
          if (c0 + 16 == half * 64 + 64) release();
          float o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = p.comp ? fmaf(a2, v2[i], a1 * v1[i]) : a1 * v1[i];
          if (store) {
            if (p.out_mode == OUT_F32) {
              float* yrow = (float*)p.y + row * p.ldy + tl.n0 + c0;
              if (p.st32) {
                st_global_32B(yrow, reinterpret_cast<const uint32_t*>(o));
                st_global_32B(yrow + 8, reinterpret_cast<const uint32_t*>(o + 8));
              } else {
                float4* dst = reinterpret_cast<float4*>(yrow);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(o[i]));
            } else {
              uint32_t packed[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                __nv_bfloat162 hb = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
                packed[i] = *reinterpret_cast<uint32_t*>(&hb);
                const float2 hr = __bfloat1622float2(hb);
                amax = fmaxf(amax, fmaxf(fabsf(hr.x), fabsf(hr.y)));
              }
              __nv_bfloat16* yrow = (__nv_bfloat16*)p.y + row * p.ldy + tl.n0 + c0;
              if (p.st32) {
                st_global_32B(yrow, packed);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(yrow);
                dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (warp == EPI_WARP0) trace_mark(p.trace, 6, j);
      if (p.y_amax) {
        amax = warp_max(amax);
        if (lane == 0 && amax > 0.0f) atomicMax(&p.y_amax[tl.e], __float_as_uint(amax));
      }
    }
  }
  // both CTAs: no MMA reads this CTA's shared memory or writes its TMEM any
  // more, and no arrival on its barriers is pending, past this point
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == MMA_WARP)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

}  // namespace pair

// ---------------------------------------------------------------- 256-column tiles
// The same product with 128 x 256 output tiles on one SM: a 256-element K
// stage is 54 KB (A 16 KB, B 32 KB, scale atoms 6 KB) and a stage's four
// 128x256x64 MMAs do twice the work of a 128x128 stage for 3/4 of its bytes,
// so the four-stage ring keeps more work in flight per byte.  The accumulator
// takes 256 TMEM columns and the scale buffers the rest, which leaves no room
// for a second accumulator: the k-channel correction is folded into the main
// one.  Its MMAs run first (the correction's stages lead each tile), the
// epilogue warps scale that partial sum by s_R / s_X in TMEM (tcgen05.ld,
// multiply, tcgen05.st), and the main MMAs then accumulate on top, so the
// epilogue forms s_X s_W (acc_main + fl(s_R / s_X * acc_corr)).
//
// Roles (24 warps):
//   warps 0-2   TMA producers (A box, B box and a scale run each; the third
//               warp two B boxes and a scale run: 18 KB per warp and stage)
//   warp 3      MMA issuer (four MMAs of a stage under one elect)
//   warps 4-7   scale atoms into TMEM: warp w the A atom and the two B atoms
//               of K step w
//   warps 8-23  epilogue: four warps per TMEM lane quadrant, 64 accumulator
//               columns each; they read their columns into registers, release
//               the accumulator, then compute and store
namespace wide {

constexpr int BM = 128, BN = 256;
constexpr int KSUB = 128;                        // bytes of a row per stage (256 FP4)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * KSUB;               // 16 KB
constexpr int B_BYTES = BN * KSUB;               // 32 KB
constexpr int OFF_B = A_BYTES;
constexpr int OFF_SFA = OFF_B + B_BYTES;         // A's atoms, one per K step
constexpr int OFF_SFB = OFF_SFA + 4 * 512;       // B rows 0-127: one atom per K step; rows 128-255 at +2 KB
constexpr int STAGE_BYTES = OFF_SFB + 8 * 512;   // 54 KB
constexpr int BOX_ROWS = 64;
constexpr int BOX_BYTES = BOX_ROWS * KSUB;       // 8 KB
constexpr int COPIES = 9;
constexpr int MMA_WARP = 3, SF_WARP0 = 4, SF_WARPS = 4, EPI_WARP0 = 8, EPI_WARPS = 16;
constexpr int NUM_THREADS = 32 * (EPI_WARP0 + EPI_WARPS);   // 768
constexpr int TMEM_COLS = 512;
constexpr int SF_COL = 256;                      // the accumulator holds columns 0-255
constexpr int SF_BUF_COLS = 48;                  // per K step q: A at 4q, B's two atoms at 16 + 8q
constexpr int SF_BUFS = 4;
static_assert(SF_COL + SF_BUFS * SF_BUF_COLS <= TMEM_COLS, "scale buffers fit beside the accumulator");
constexpr int MAX_GROUPS = 256;
constexpr int BAR_BYTES = 1024;
constexpr int META_BYTES = 4 * (MAX_GROUPS + 1) + 3 * 4 * MAX_GROUPS;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + META_BYTES + 1024 /*align*/;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

struct Meta {
  int32_t* off;    // [E+1]
  int32_t* cnt;    // [E]
  float* a1;       // [E] s_a * s_w
  float* ratio;    // [E] s_r / s_a
};

__device__ __forceinline__ int64_t total_tiles(const Params& p, const Meta& m) {
  if (!p.row_off) return ((p.M + BM - 1) / BM) * p.Nt;
  return (int64_t)(m.off[p.E] / BM) * p.Nt;
}

__device__ __forceinline__ Tile decode_tile(const Params& p, const Meta& m, int64_t t) {
  Tile r;
  if (!p.row_off) {
    const int64_t Mt = (p.M + BM - 1) / BM;
    r.e = 0;
    r.m0 = (t % Mt) * BM;
    r.n0 = (int)(t / Mt) * BN;
    r.row_end = p.M;
    return r;
  }
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)(m.off[mid] / BM) * p.Nt <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int64_t base = (int64_t)(m.off[e] / BM) * p.Nt;
  const int64_t mt_e = (m.off[e + 1] - m.off[e]) / BM;
  const int64_t local = t - base;
  r.e = e;
  r.m0 = m.off[e] + (local % mt_e) * BM;
  r.n0 = (int)(local / mt_e) * BN;
  r.row_end = m.off[e] + m.cnt[e];
  return r;
}

// Stage j of a tile: the correction's stages first, then the main range's.
struct Stage {
  int ksteps;
  bool corr;
  int kk;       // stage index inside its own K range
};
__device__ __forceinline__ Stage stage_of(const Params& p, int j, int ncorr) {
  Stage s;
  s.corr = j < ncorr;
  s.kk = s.corr ? j : j - ncorr;
  s.ksteps = min(4, ((s.corr ? p.kpad : p.K) - s.kk * 256) / 64);
  return s;
}

// Four 128x256x64 MMAs of a stage under one elect: descriptors +2 per K
// step, A's scale columns +4, B's +8.
__device__ __forceinline__ void mma_x4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 a1, b1;\n\t.reg .b32 fa, fb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\tadd.u32 fa, %5, 4;\n\tadd.u32 fb, %6, 8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\tadd.u32 fa, %5, 8;\n\tadd.u32 fb, %6, 16;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\tadd.u32 fa, %5, 12;\n\tadd.u32 fb, %6, 24;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [fa], [fb], 1;\n\t"
      "}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}

// K step q's atoms: A to column t, B rows 0-127 to t + 16 + 4q... (caller
// passes both targets), under one elect.
__device__ __forceinline__ void cp_atoms3(uint32_t ta, uint64_t da, uint32_t tb, uint64_t db0,
                                          uint64_t db1) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 t1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "add.u32 t1, %2, 4;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%2], %3;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [t1], %4;\n\t}" ::"r"(ta),
      "l"(da), "r"(tb), "l"(db0), "l"(db1)
      : "memory");
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    wide_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmW,
                     const Params p) {
  griddep_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;                           // [STAGES]
  uint64_t* empty = full + STAGES;                 // [STAGES]
  uint64_t* sf_ready = empty + STAGES;             // [SF_BUFS]
  uint64_t* acc_full = sf_ready + SF_BUFS;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* corr_full = acc_empty + 1;
  uint64_t* prescaled = corr_full + 1;
  uint64_t* drain_mma = prescaled + 1;
  uint64_t* drain_sf = drain_mma + 1;
  uint32_t* tmem_holder = (uint32_t*)(drain_sf + 1);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  Meta meta;
  meta.off = (int32_t*)(smem + STAGES * STAGE_BYTES + BAR_BYTES);
  meta.cnt = meta.off + (MAX_GROUPS + 1);
  meta.a1 = (float*)(meta.cnt + MAX_GROUPS);
  meta.ratio = meta.a1 + MAX_GROUPS;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const float ats = __ldg(p.a_ts + (p.a_ts_pe ? e : 0));
    meta.a1[e] = __fmul_rn(ats, __ldg(p.b_ts + e));
    meta.ratio[e] = p.comp ? __fdiv_rn(__ldg(p.r_ts + (p.r_ts_pe ? e : 0)), ats) : 0.0f;
    if (p.row_off) {
      meta.off[e] = p.row_off[e];
      meta.cnt[e] = p.row_cnt ? p.row_cnt[e] : (p.row_off[e + 1] - p.row_off[e]);
    }
  }
  if (threadIdx.x == 0 && p.row_off) meta.off[p.E] = p.row_off[p.E];
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) { mbar_init(&full[i], COPIES); mbar_init(&empty[i], 1); }
    for (int i = 0; i < SF_BUFS; ++i) mbar_init(&sf_ready[i], SF_WARPS);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, EPI_WARPS);
    mbar_init(corr_full, 1);
    mbar_init(prescaled, EPI_WARPS);
    mbar_init(drain_mma, 1);
    mbar_init(drain_sf, SF_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const Sync sy{abort_flag, p.err, p.timeout_ns};
  const Sync dr{abort_flag, p.err, kDrainNs};

  const int64_t ntiles = total_tiles(p, meta);
  const int nmain = (p.K + 255) / 256;
  const int ncorr = p.comp ? (p.kpad + 255) / 256 : 0;
  const int nst = ncorr + nmain;
  const int64_t a_sf_rb = (int64_t)(p.K / 64) * 512;   // scale bytes per 128-row block
  const int64_t r_sf_rb = (int64_t)(p.kpad / 64) * 512;

  if (warp < 3) {
    // ------------------------------------------------------------ producers
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const Tile tl = decode_tile(p, meta, t);
      const int64_t brow = (int64_t)tl.e * p.N + tl.n0;
      for (int j = 0; j < nst && ok; ++j, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        const Stage sg = stage_of(p, j, ncorr);
        uint8_t* st = smem + s * STAGE_BYTES;
        if (!warp_wait(&empty[s], ph ^ 1, sy)) { ok = false; break; }
        if (warp == 0) trace_mark(p.trace, 0, it);
        if (elect_one()) {
          const int x = sg.kk * KSUB;
          const CUtensorMap* ma = sg.corr ? &tmR : &tmA;
          const CUtensorMap* mb = sg.corr ? &tmW : &tmB;
          const int64_t rb = sg.corr ? r_sf_rb : a_sf_rb;
          const uint32_t sfbytes = sg.ksteps * 512;
          // warp 0: A rows 0-63, B rows 0-63, A's atoms; warp 1: A rows 64-127,
          // B rows 64-127, B's atoms of rows 0-127; warp 2: B rows 128-255 and
          // their atoms
          for (int c = 0; c < 3; ++c) {
            const int kind = warp == 2 ? (c < 2 ? 1 : 2) : c;   // 0: A box, 1: B box, 2: atoms
            if (kind == 0) {
              mbar_expect_tx(&full[s], BOX_BYTES);
              tma_load_2d(st + warp * BOX_BYTES, ma, x, (int)(tl.m0 + warp * BOX_ROWS), &full[s]);
            } else if (kind == 1) {
              const int bb = warp == 2 ? 2 + c : warp;
              mbar_expect_tx(&full[s], BOX_BYTES);
              tma_load_2d(st + OFF_B + bb * BOX_BYTES, mb, x, (int)(brow + bb * BOX_ROWS), &full[s]);
            } else {
              const uint8_t* base = warp == 0 ? (sg.corr ? p.r_sf : p.a_sf) : (sg.corr ? p.ws_sf : p.b_sf);
              const int64_t blk = warp == 0 ? tl.m0 / BM : brow / BM + (warp == 2 ? 1 : 0);
              const uint8_t* src = base + blk * rb + (int64_t)sg.kk * 2048;
              [[maybe_unused]] const int64_t lim = warp == 0 ? (sg.corr ? p.r_sf_bytes : p.a_sf_bytes)
                                                              : (sg.corr ? p.ws_sf_bytes : p.b_sf_bytes);
              if (!QDBGV(src - base + sfbytes <= lim,
                         (tl.m0 << 20) | ((int64_t)tl.e << 8) | (sg.corr ? 2 : 0) | warp)) {
                mbar_arrive(&full[s]);   // skipped copy: the stage still completes
                continue;
              }
              mbar_expect_tx(&full[s], sfbytes);
              bulk_load(st + (warp == 0 ? OFF_SFA : OFF_SFB + (warp == 2 ? 2048 : 0)), src, sfbytes,
                        &full[s]);
            }
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      // the copies this warp issued land before the CTA can exit (a fixed
      // bounded time: a stage's barrier may never complete once another
      // producer stopped before its share)
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < kCopyDrainNs) {
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_nvf4(BM, BN);
    uint32_t s = 0, sb = 0, sph = 0, mit = 0;
    uint32_t j = 0;
    bool ok = !p.skip_mma;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++j) {
      // the epilogue has read the previous tile's accumulator
      if (!conv_wait(acc_empty, (j & 1) ^ 1, sy)) { ok = false; break; }
      tc_fence_after();
      for (int q = 0; q < nst; ++q) {
        const Stage sg = stage_of(p, q, ncorr);
        if (q == ncorr && ncorr > 0) {
          // the correction's partial sum is complete: the epilogue scales it
          // by s_R / s_X in place before the main range accumulates on top
          tc_commit_el(corr_full);
          if (!conv_wait(prescaled, j & 1, sy)) { ok = false; break; }
          tc_fence_after();
        }
        if (!conv_wait(&sf_ready[sb], sph, sy)) { ok = false; break; }
        trace_mark(p.trace, 3, mit);
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
        const uint32_t tsf = tmem + SF_COL + sb * SF_BUF_COLS;
        // accumulate onto earlier stages, the prescaled correction included
        const uint32_t acc = (q > 0) ? 1u : 0u;
        if (sg.ksteps == 4) {
          mma_x4(tmem, desc_sw128(sa), desc_sw128(sa + OFF_B), idesc, tsf, tsf + 16, acc);
        } else {
          for (int k = 0; k < sg.ksteps; ++k)
            tc_mma_el(tmem, desc_sw128(sa + 32 * k), desc_sw128(sa + OFF_B + 32 * k), idesc,
                      tsf + 4 * k, tsf + 16 + 8 * k, (acc || k > 0) ? 1u : 0u);
        }
        tc_commit_el(&empty[s]);   // also frees this stage's scale buffer
        trace_mark(p.trace, 4, mit++);
        if (++s == STAGES) s = 0;
        if (++sb == SF_BUFS) { sb = 0; sph ^= 1; }
      }
      if (!ok) break;
      tc_commit_el(acc_full);
    }
    tc_commit_el(drain_mma);
    if (lane == 0) wait1(drain_mma, 0, dr, false, true);
    __syncwarp();
  } else if (warp >= SF_WARP0 && warp < EPI_WARP0) {
    // ------------------------------------------------------------ scale staging
    // TMEM buffer sb: K step q's A atom at column SF_COL + 48*sb + 4q, B's
    // atoms of rows 0-127 and 128-255 at +16 + 8q and +20 + 8q (row r of an
    // operand at lane r % 32, column r / 32, as the block-scaled MMA reads
    // them).  Warp w copies K step w's three atoms once the stage has landed;
    // buffer sb was last read by the MMAs of ring iteration it - SF_BUFS.
    const int w = warp - SF_WARP0;
    uint32_t s = 0, ph = 0, sb = 0, it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      for (int q = 0; q < nst; ++q, ++it) {
        bool okw = conv_wait(&full[s], ph, sy);
        if (okw && it >= (uint32_t)SF_BUFS) {
          const uint32_t prev = it - SF_BUFS;
          okw = conv_wait(&empty[prev % STAGES], (prev / STAGES) & 1, sy);
        }
        if (!okw) { ok = false; break; }
        if (w == 0) trace_mark(p.trace, 1, it);
        tc_fence_after();
        const Stage sg = stage_of(p, q, ncorr);
        if (w < sg.ksteps) {
          const uint32_t ss = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t tsf = tmem + SF_COL + sb * SF_BUF_COLS;
          cp_atoms3(tsf + 4 * w, desc_sf(ss + OFF_SFA + 512 * w), tsf + 16 + 8 * w,
                    desc_sf(ss + OFF_SFB + 512 * w), desc_sf(ss + OFF_SFB + 2048 + 512 * w));
        }
        tc_commit_el(&sf_ready[sb]);
        if (w == 0) trace_mark(p.trace, 2, it);
        if (++s == STAGES) { s = 0; ph ^= 1; }
        if (++sb == SF_BUFS) sb = 0;
      }
    }
    tc_commit_el(drain_sf);
    if (lane == 0) wait1(drain_sf, 0, dr, false, true);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - EPI_WARP0;
    const int quad = warp & 3;               // TMEM lane quadrant this warp may access
    const int sub = ew >> 2;                 // which 64 of the tile's 256 columns
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const bool swiglu = p.out_mode == OUT_SWIGLU;
    // this warp's accumulator columns: SwiGLU: 32 gate columns and the
    // matching 32 up columns (tile columns [128b, 128b + 64) are gate rows of
    // W, the next 64 the up rows); otherwise 64 consecutive columns
    const int c_lo = swiglu ? 128 * (sub >> 1) + 32 * (sub & 1) : 64 * sub;
    const int c_hi = swiglu ? c_lo + 64 : c_lo + 32;   // second half of the 64
    uint32_t j = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
      const Tile tl = decode_tile(p, meta, t);
      if (p.comp) {
        if (!warp_wait(corr_full, j & 1, sy)) break;
        tc_fence_after();
        // all four loads, one wait, all four stores, one wait
        const float ratio = meta.ratio[tl.e];
        float w[64];
        tc_ld16(tmem + lane_base + c_lo, w);
        tc_ld16(tmem + lane_base + c_lo + 16, w + 16);
        tc_ld16(tmem + lane_base + c_hi, w + 32);
        tc_ld16(tmem + lane_base + c_hi + 16, w + 48);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 64; ++i) w[i] = __fmul_rn(ratio, w[i]);
        tc_st16(tmem + lane_base + c_lo, w);
        tc_st16(tmem + lane_base + c_lo + 16, w + 16);
        tc_st16(tmem + lane_base + c_hi, w + 32);
        tc_st16(tmem + lane_base + c_hi + 16, w + 48);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(prescaled);
      }
      if (!warp_wait(acc_full, j & 1, sy)) break;
      if (warp == EPI_WARP0) trace_mark(p.trace, 5, j);
      tc_fence_after();
      float v[64];
      tc_ld16(tmem + lane_base + c_lo, v);
      tc_ld16(tmem + lane_base + c_lo + 16, v + 16);
      tc_ld16(tmem + lane_base + c_hi, v + 32);
      tc_ld16(tmem + lane_base + c_hi + 16, v + 48);
      tc_wait_ld();
      // the accumulator is read: release it before the math and the stores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      const float a1 = meta.a1[tl.e];
      const int64_t row = tl.m0 + row_in_tile;
      float amax = 0.0f;
      if (swiglu) {
        const bool store = row < (p.row_off ? (int64_t)meta.off[tl.e + 1] : p.M) && QDBG(row < p.y_rows);
        // v[0..31]: gate columns, v[32..63]: the matching up columns
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float h[2];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float g = a1 * v[i + q], u = a1 * v[32 + i + q];
            h[q] = __fdividef(g * u, 1.0f + __expf(-g));   // silu(g) * u
          }
          __nv_bfloat162 hb = __floats2bfloat162_rn(h[0], h[1]);
          packed[i / 2] = *reinterpret_cast<uint32_t*>(&hb);
          const float2 hr = __bfloat1622float2(hb);
          amax = fmaxf(amax, fmaxf(fabsf(hr.x), fabsf(hr.y)));
        }
        if (store) {
          __nv_bfloat16* y = (__nv_bfloat16*)p.y + row * p.ldy + tl.n0 / 2 + 64 * (sub >> 1) + 32 * (sub & 1);
          if (p.st32) {
            st_global_32B(y, packed);
            st_global_32B(y + 16, packed + 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(y);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
          }
        } else {
          amax = 0.0f;
        }
      } else {
        const bool store = row < tl.row_end && QDBG(row < p.y_rows);
        if (store) {
          if (p.out_mode == OUT_F32) {
            float* yrow = (float*)p.y + row * p.ldy + tl.n0 + 64 * sub;
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = a1 * v[i];
            if (p.st32) {
#pragma unroll
              for (int i = 0; i < 8; ++i) st_global_32B(yrow + 8 * i, reinterpret_cast<const uint32_t*>(v + 8 * i));
            } else {
              float4* dst = reinterpret_cast<float4*>(yrow);
#pragma unroll
              for (int i = 0; i < 16; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
          } else {
            uint32_t packed[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              __nv_bfloat162 hb = __floats2bfloat162_rn(a1 * v[2 * i], a1 * v[2 * i + 1]);
              packed[i] = *reinterpret_cast<uint32_t*>(&hb);
              const float2 hr = __bfloat1622float2(hb);
              amax = fmaxf(amax, fmaxf(fabsf(hr.x), fabsf(hr.y)));
            }
            __nv_bfloat16* yrow = (__nv_bfloat16*)p.y + row * p.ldy + tl.n0 + 64 * sub;
            if (p.st32) {
#pragma unroll
              for (int i = 0; i < 4; ++i) st_global_32B(yrow + 16 * i, packed + 8 * i);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(yrow);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
            }
          }
        }
      }
      __syncwarp();
      if (warp == EPI_WARP0) trace_mark(p.trace, 6, j);
      if (p.y_amax) {
        amax = warp_max(amax);
        if (lane == 0 && amax > 0.0f) atomicMax(&p.y_amax[tl.e], __float_as_uint(amax));
      }
    }
  }
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

}  // namespace wide

// ---------------------------------------------------------------- Q(W_sel)
// Column-major copy of an NVFP4 weight, made once per weight update: for group
// g (rows g*N .. g*N+N-1), codes_t[g][c][n/2] holds the codes of rows n, n+1 at
// column c (n even -> low nibble) and scales_t[g][c/16][n] the block scale, so
// the k selected columns are read as k contiguous runs.
// One CTA per (group, 128-row block, 64-column group): the block's codes
// (128 rows x 32 bytes) are staged in shared memory and written back as 64
// columns x 64 bytes; the block's one scale atom (128 rows x 4 scale columns,
// 512 contiguous bytes) becomes 4 scale rows of 128 bytes.  Every global
// access is a coalesced run.
__global__ void __launch_bounds__(256) wtrans_kernel(const uint8_t* __restrict__ wc,
                                                     const uint8_t* __restrict__ wsf, int G, int N,
                                                     int K, uint8_t* __restrict__ ct,
                                                     uint8_t* __restrict__ st) {
  __shared__ __align__(16) uint8_t tile[128][32];
  const int ncg = K / 64, nrb = N / 128;
  const int64_t id = blockIdx.x;
  const int cg = (int)(id % ncg);
  const int rb = (int)((id / ncg) % nrb);
  const int g = (int)(id / ((int64_t)ncg * nrb));
  const int t = threadIdx.x;
  const int64_t row0 = (int64_t)g * N + (int64_t)rb * 128;   // first weight row of the block
  {
    const int r = t >> 1, h = t & 1;
    reinterpret_cast<uint4*>(tile[r])[h] =
        __ldg(reinterpret_cast<const uint4*>(wc + (row0 + r) * (K / 2) + cg * 32) + h);
  }
  __syncthreads();
  {
    const int cc = t >> 2, part = t & 3;           // column cg*64 + cc, row pairs part*16 ..
    const uint32_t sh = (cc & 1) * 4;
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int np = part * 16 + i;
      const uint32_t lo = (tile[2 * np][cc >> 1] >> sh) & 15u;
      const uint32_t hi = (tile[2 * np + 1][cc >> 1] >> sh) & 15u;
      w[i >> 2] |= (lo | (hi << 4)) << (8 * (i & 3));
    }
    uint8_t* dst = ct + (int64_t)g * K * (N / 2) + (int64_t)(cg * 64 + cc) * (N / 2) + rb * 64 + part * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (t < 128) {
    const uint8_t* atom = wsf + ((row0 / 128) * (K / 64) + cg) * 512;
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(atom + (t & 31) * 16 + ((t >> 5) & 3) * 4));
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st[((int64_t)g * (K / 16) + cg * 4 + j) * N + rb * 128 + t] = (uint8_t)(v >> (8 * j));
  }
}

// Q(W_sel): for every weight row r (of every expert) and every 16-block of the
// selected channels, gather the selected columns of DQ(Q(W)) in units of s_w
// (level * E4M3 scale, exact) and requantize with tensor scale 1 (s_w kept).
// Output codes [E*N, kpad/2] and TCGEN05 scales over kpad columns.
// One CTA per (16-column block of the selection, group, chunk of NC rows):
// the chunk's codes (NC/2 bytes) and scale bytes (NC) of
// the block's 16 selected columns -- contiguous runs in the column-major copy
// -- are staged in shared memory with 16-byte loads, then each thread
// requantizes rows from there.  Long runs keep DRAM and L2 busy, where
// per-row 16/32-byte gathers wait on latency.  Padding blocks (>= k) get zero
// codes and scales.
__global__ void __launch_bounds__(256) wsel_cols_kernel(
    const uint8_t* __restrict__ ct, const uint8_t* __restrict__ st, int N, int K, int NC,
    const int32_t* __restrict__ sel, int sel_pe, int k, int kpad, uint8_t* __restrict__ oc,
    uint8_t* __restrict__ osf) {
  griddep_wait();
  extern __shared__ __align__(16) uint8_t wsm[];
  uint8_t* sc = wsm;                   // [16][NC/2] codes
  uint8_t* ss = wsm + 16 * (NC / 2);   // [16][NC] scale bytes
  const int blk = blockIdx.x, e = blockIdx.y, n0 = blockIdx.z * NC, nb = kpad >> 4;
  const int64_t r0 = (int64_t)e * N + n0;
  if (blk * 16 >= k) {
    for (int n = threadIdx.x; n < NC; n += blockDim.x) {
      *reinterpret_cast<uint2*>(oc + (r0 + n) * (kpad >> 1) + blk * 8) = make_uint2(0, 0);
      osf[sf_tc_offset(r0 + n, blk, nb)] = 0;
    }
    return;
  }
  const int32_t* s = sel + (sel_pe ? (int64_t)e * k : 0) + blk * 16;
  const uint8_t* cte = ct + (int64_t)e * K * (N / 2) + n0 / 2;
  const uint8_t* ste = st + (int64_t)e * (K / 16) * N + n0;
  const int cv = NC >> 5, sv = NC >> 4;   // 16-byte vectors per code run / scale run
  for (int i = threadIdx.x; i < 16 * (cv + sv); i += blockDim.x) {
    if (i < 16 * cv) {
      const int j = i / cv, v = i - j * cv;
      int c = __ldg(s + j);
      if (!QDBG(c >= 0 && c < K)) c = 0;
      reinterpret_cast<uint4*>(sc + j * (NC / 2))[v] =
          __ldg(reinterpret_cast<const uint4*>(cte + (int64_t)c * (N / 2)) + v);
    } else {
      const int i2 = i - 16 * cv, j = i2 / sv, v = i2 - j * sv;
      int c = __ldg(s + j);
      if (!QDBG(c >= 0 && c < K)) c = 0;
      reinterpret_cast<uint4*>(ss + j * NC)[v] =
          __ldg(reinterpret_cast<const uint4*>(ste + (int64_t)(c >> 4) * N) + v);
    }
  }
  __syncthreads();
  for (int n = threadIdx.x; n < NC; n += blockDim.x) {
    const uint32_t sh = (n & 1) * 4;
    // two columns at a time: level x E4M3 value is exact in f16 (at most 6
    // significant bits, magnitudes 2^-10 .. 2688), so packed f16x2 decodes and
    // one HMUL2 give the same values as float32 products
    float w16[16];
    __half2 m2 = __float2half2_rn(0.0f);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int j = 2 * p;
      const uint32_t c2 = ((sc[j * (NC / 2) + (n >> 1)] >> sh) & 15u) |
                          (((sc[(j + 1) * (NC / 2) + (n >> 1)] >> sh) & 15u) << 4);
      const uint32_t s2 = (uint32_t)ss[j * NC + n] | ((uint32_t)ss[(j + 1) * NC + n] << 8);
      uint32_t lv, sv;
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b16 lo;\n\t"
          "mov.b32 {b0, b1, b2, b3}, %2;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
          "cvt.u16.u32 lo, %3;\n\t"
          "cvt.rn.f16x2.e4m3x2 %1, lo;\n\t}"
          : "=r"(lv), "=r"(sv)
          : "r"(c2), "r"(s2));
      const __half2 w = __hmul2(*reinterpret_cast<const __half2*>(&lv),
                                *reinterpret_cast<const __half2*>(&sv));
      m2 = __hmax2(m2, __habs2(w));
      const float2 wf = __half22float2(w);
      w16[j] = wf.x;
      w16[j + 1] = wf.y;
    }
    const float2 mf = __half22float2(m2);
    const BlockScale bs = block_scale(fmaxf(mf.x, mf.y), 1.0f);
    *reinterpret_cast<uint2*>(oc + (r0 + n) * (kpad >> 1) + blk * 8) =
        make_uint2(quantize8(w16, bs), quantize8(w16 + 8, bs));
    osf[sf_tc_offset(r0 + n, blk, nb)] = (uint8_t)bs.byte;
  }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
  }
  return fn;
}

// 2-D byte tensor [rows, width_bytes] (row pitch ld_bytes), box 128 B x 64 rows,
// 128-byte swizzle, out-of-range elements read as zero.
static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t width_bytes,
                     int64_t ld_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld_bytes};
  cuuint32_t box[2] = {KSUB, BOX_ROWS};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Scale atoms as rows of 128 bytes (a 512-byte atom is four rows), box of
// `box_rows` rows, no swizzle: the pair kernel loads a sub-tile's atoms with
// one TMA copy that can complete on the leader CTA's barrier.
static bool make_sf_map(CUtensorMap* m, const void* base, int64_t bytes, int box_rows) {
  auto fn = encode_fn();
  if (!fn || bytes < 128 || bytes % 128) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)(bytes / 128)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static __device__ int g_gemm_error;

// Test hook (quads_test_gemm_wait_timeout): the next GEMM launch gets a 1 ms
// wait limit and an MMA warp that issues nothing, so its waits run out.
static std::atomic<int> g_wait_test{0};
// Profiling hook (quads_test_gemm_timeline): the next one-CTA GEMM launch
// records CTA 0's stage timeline into this device buffer.
static std::atomic<unsigned long long*> g_trace{nullptr};
// The CTA-pair kernel, selectable for comparison (QUADS_GEMM_PAIR=1); the
// one-CTA kernel measured faster on every benchmark shape and is the default.
// Tile width policy (quads_set_gemm_tile_policy).
static std::atomic<int> g_tile_policy{QUADS_GEMM_TILES_AUTO};
static const bool g_pair_kernel = [] {
  const char* v = getenv("QUADS_GEMM_PAIR");
  return v && v[0] == '1';
}();

struct Launch {
  int64_t M, rows_cap;
  int E, N, K, k, kpad;
  const int32_t* row_off;
  const int32_t* row_cnt;
  const uint8_t *a, *a_sf, *b, *b_sf, *b_t, *b_sf_t, *r, *r_sf;
  const uint8_t *wsel, *wsel_sf;   // prebuilt Q(W_sel), or null: built into ws
  const float *a_ts, *b_ts, *r_ts;
  int a_pe, r_pe;
  const int32_t* sel;
  int sel_pe;
  void* y;
  int64_t ldy;
  int out_mode;
  int mx;
  float* y_amax;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
};

// Q(W_sel) of E groups of N rows: codes [E*N, kpad/2], TCGEN05 scales.
static void launch_wsel(const uint8_t* b_t, const uint8_t* b_sf_t, int E, int N, int K,
                        const int32_t* sel, int sel_pe, int k, int kpad, uint8_t* codes,
                        uint8_t* sf, cudaStream_t stream) {
  // rows per CTA: the largest chunk (N is a multiple of 128) that still
  // gives every SM work and fits one resident wave (eight CTAs per SM), so
  // that no partial second wave doubles the time; else 128-row chunks
  const int64_t per_chunk = (int64_t)(kpad / 16) * E;
  int NC = 128;
  for (const int c : {1024, 768, 512, 256}) {
    const int64_t ctas = per_chunk * (N / c);
    if (N % c == 0 && ctas >= num_sms() && ctas <= 8 * (int64_t)num_sms()) {
      NC = c;
      break;
    }
  }
  const size_t cols_smem = (size_t)24 * NC;   // 16 columns x (NC/2 code + NC scale bytes)
  const dim3 grid((unsigned)(kpad / 16), (unsigned)E, (unsigned)(N / NC));
  launch_dep(wsel_cols_kernel, grid, 256, cols_smem, stream, b_t, b_sf_t, N, K, NC, sel, sel_pe, k,
             kpad, codes, sf);
}

static quads_status_t launch(const Launch& L) {
  const bool comp = L.r != nullptr;
  const int64_t brows = (int64_t)L.E * L.N;
  const uint8_t* ws_codes = nullptr;
  const uint8_t* ws_sf = nullptr;
  int launches = comp ? 2 : 1;
  if (comp && L.wsel) {
    ws_codes = L.wsel;
    ws_sf = L.wsel_sf;
    launches = 1;
  } else if (comp) {
    const size_t need = quads_workspace_size(L.row_off ? QUADS_OP_MOE_GEMM : QUADS_OP_GEMM, 0,
                                             L.K, L.N, L.k, L.E);
    if (!L.ws || L.ws_bytes < need)
      return fail(QUADS_ERR_WORKSPACE, "gemm: workspace needs %zu bytes", need);
    if ((uintptr_t)L.ws & 15u) return fail(QUADS_ERR_MISALIGNED, "gemm: workspace must be 16-byte aligned");
    uint8_t* c = (uint8_t*)L.ws;
    uint8_t* f = c + (((size_t)brows * (L.kpad / 2) + 1023) & ~(size_t)1023);
    launch_wsel(L.b_t, L.b_sf_t, L.E, L.N, L.K, L.sel, L.sel_pe, L.k, L.kpad, c, f, L.stream);
    ws_codes = c;
    ws_sf = f;
  }
  CUtensorMap tA, tB, tR, tW;
  const int64_t arows = L.row_off ? L.rows_cap : L.M;
  if (!make_map(&tA, L.a, arows, L.K / 2, L.K / 2) || !make_map(&tB, L.b, brows, L.K / 2, L.K / 2))
    return fail(QUADS_ERR_CUDA, "gemm: cuTensorMapEncodeTiled failed for A/W");
  if (comp) {
    if (!make_map(&tR, L.r, arows, L.kpad / 2, L.kpad / 2) ||
        !make_map(&tW, ws_codes, brows, L.kpad / 2, L.kpad / 2))
      return fail(QUADS_ERR_CUDA, "gemm: cuTensorMapEncodeTiled failed for R/W_sel");
  } else {
    tR = tA;
    tW = tB;
  }
  // 32-byte stores need every row start and column offset on a 32-byte
  // boundary: tiles start at multiples of 128 columns (64 for SwiGLU output)
  const int64_t esz = L.out_mode == OUT_F32 ? 4 : 2;
  const int st32 = ((uintptr_t)L.y % 32 == 0 && (L.ldy * esz) % 32 == 0) ? 1 : 0;
  // scale buffer sizes implied by the shapes (checked in bounds-checked builds)
  struct { int64_t a, b, r, w; } ext;
  {
    const int64_t per = L.mx ? 32 : 16;
    ext.a = (arows + 127) / 128 * 128 * (L.K / per);
    ext.b = (brows + 127) / 128 * 128 * (L.K / per);
    ext.r = comp ? (arows + 127) / 128 * 128 * (L.kpad / 16) : 0;
    ext.w = comp ? (brows + 127) / 128 * 128 * (L.kpad / 16) : 0;
  }
  if (L.y_amax) cudaMemsetAsync(L.y_amax, 0, (size_t)L.E * 4, L.stream);
  // per device, resolved on the first launch there (calls after
  // cudaDeviceReset are not supported): the error word's address, the
  // shared-memory attributes and how many CTA pairs can be resident at once
  int* errp = nullptr;
  int max_pairs = 0;
  {
    static std::mutex mu;
    static int* errp_dev[64] = {nullptr};
    static int pairs_dev[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
      return fail(QUADS_ERR_CUDA, "gemm: no usable current device (ordinal %d)", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!errp_dev[dev]) {
      if (cudaGetSymbolAddress((void**)&errp_dev[dev], g_gemm_error) != cudaSuccess) {
        errp_dev[dev] = nullptr;
        return fail(QUADS_ERR_CUDA, "gemm: cannot resolve the device error word");
      }
      cudaError_t e = cudaFuncSetAttribute(gemm_kernel<Geo512>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Geo512::SMEM_BYTES);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_kernel<Geo256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Geo256::SMEM_BYTES);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(pair::pair_gemm_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pair::SMEM_BYTES);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(wide::wide_gemm_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, wide::SMEM_BYTES);
      if (e != cudaSuccess) {
        errp_dev[dev] = nullptr;
        return fail(QUADS_ERR_CUDA, "gemm: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      }
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 2;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (unsigned)num_sms(), 1, 1);
      cfg.blockDim = dim3(pair::NUM_THREADS, 1, 1);
      cfg.dynamicSmemBytes = pair::SMEM_BYTES;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, pair::pair_gemm_kernel, &cfg);
      if (e != cudaSuccess || n < 1) {
        errp_dev[dev] = nullptr;
        return fail(QUADS_ERR_CUDA, "gemm: no resident CTA pair possible (%s)",
                    e == cudaSuccess ? "0 clusters" : cudaGetErrorString(e));
      }
      pairs_dev[dev] = n;
    }
    errp = errp_dev[dev];
    max_pairs = pairs_dev[dev];
  }
  const bool wait_test = g_wait_test.exchange(0) != 0;
  const int policy = g_tile_policy.load();
  if (!g_pair_kernel && !L.mx && L.N % wide::BN == 0 &&
      (policy == QUADS_GEMM_TILES_256 || (policy == QUADS_GEMM_TILES_AUTO && !comp))) {
    Params p;
    p.E = L.E; p.N = L.N; p.K = L.K; p.kpad = comp ? L.kpad : 0; p.Nt = L.N / wide::BN;
    p.M = L.M; p.row_off = L.row_off; p.row_cnt = L.row_cnt;
    p.a_sf = L.a_sf; p.b_sf = L.b_sf; p.r_sf = L.r_sf; p.ws_sf = ws_sf;
    p.a_ts = L.a_ts; p.b_ts = L.b_ts; p.r_ts = L.r_ts; p.a_ts_pe = L.a_pe; p.r_ts_pe = L.r_pe;
    p.comp = comp ? 1 : 0;
    p.mx = 0;
    p.y = L.y; p.ldy = L.ldy; p.out_mode = L.out_mode;
    p.st32 = st32;
    p.y_amax = (uint32_t*)L.y_amax;
    p.err = errp;
    p.a_sf_bytes = ext.a; p.b_sf_bytes = ext.b; p.r_sf_bytes = ext.r; p.ws_sf_bytes = ext.w;
    p.y_rows = arows;
    p.timeout_ns = wait_test ? 1000000ull : kTimeoutNs;
    p.skip_mma = wait_test ? 1 : 0;
    p.trace = g_trace.exchange(nullptr);
    int64_t grid = num_sms();
    if (!L.row_off) grid = std::min<int64_t>(grid, ((L.M + wide::BM - 1) / wide::BM) * p.Nt);
    launch_dep(wide::wide_gemm_kernel, (int)grid, wide::NUM_THREADS, wide::SMEM_BYTES, L.stream,
        tA, tB, tR, tW, p);
    return check_launch("gemm", launches);
  }
  if (!g_pair_kernel) {
    Params p;
    p.E = L.E; p.N = L.N; p.K = L.K; p.kpad = comp ? L.kpad : 0; p.Nt = L.N / BN;
    p.M = L.M; p.row_off = L.row_off; p.row_cnt = L.row_cnt;
    p.a_sf = L.a_sf; p.b_sf = L.b_sf; p.r_sf = L.r_sf; p.ws_sf = ws_sf;
    p.a_ts = L.a_ts; p.b_ts = L.b_ts; p.r_ts = L.r_ts; p.a_ts_pe = L.a_pe; p.r_ts_pe = L.r_pe;
    p.comp = comp ? 1 : 0;
    p.mx = L.mx;
    p.y = L.y; p.ldy = L.ldy; p.out_mode = L.out_mode;
    p.st32 = st32;
    p.y_amax = (uint32_t*)L.y_amax;
    p.err = errp;
    p.a_sf_bytes = ext.a; p.b_sf_bytes = ext.b; p.r_sf_bytes = ext.r; p.ws_sf_bytes = ext.w;
    p.y_rows = arows;
    p.timeout_ns = wait_test ? 1000000ull : kTimeoutNs;
    p.skip_mma = wait_test ? 1 : 0;
    p.trace = g_trace.exchange(nullptr);
    int64_t grid = num_sms();
    if (!L.row_off) grid = std::min<int64_t>(grid, ((L.M + BM - 1) / BM) * (L.N / BN));
    // 256-element stages when K leaves a 512-element ring with a half-empty stage
    if (L.K % 512)
      launch_dep(gemm_kernel<Geo256>, (int)grid, NUM_THREADS, Geo256::SMEM_BYTES, L.stream,
          tA, tB, tR, tW, p);
    else
      launch_dep(gemm_kernel<Geo512>, (int)grid, NUM_THREADS, Geo512::SMEM_BYTES, L.stream,
          tA, tB, tR, tW, p);
    return check_launch("gemm", launches);
  }
  pair::Params p;
  p.E = L.E; p.N = L.N; p.K = L.K; p.kpad = comp ? L.kpad : 0; p.Nt = L.N / pair::BN;
  p.M = L.M; p.row_off = L.row_off; p.row_cnt = L.row_cnt;
  p.a_sf = L.a_sf; p.b_sf = L.b_sf; p.r_sf = L.r_sf; p.ws_sf = ws_sf;
  p.a_ts = L.a_ts; p.b_ts = L.b_ts; p.r_ts = L.r_ts; p.a_ts_pe = L.a_pe; p.r_ts_pe = L.r_pe;
  p.comp = comp ? 1 : 0;
  p.mx = L.mx;
  p.y = L.y; p.ldy = L.ldy; p.out_mode = L.out_mode;
  p.st32 = st32;
  p.y_amax = (uint32_t*)L.y_amax;
  p.err = errp;
  p.a_sf_bytes = ext.a; p.b_sf_bytes = ext.b; p.r_sf_bytes = ext.r; p.ws_sf_bytes = ext.w;
  p.y_rows = arows;
  p.timeout_ns = wait_test ? 1000000ull : kTimeoutNs;
  p.skip_mma = wait_test ? 1 : 0;
  p.trace = g_trace.exchange(nullptr);
  // one CTA pair per pair of SMs, persistent over the tiles
  int64_t pairs = max_pairs;
  if (!L.row_off)
    pairs = std::min<int64_t>(pairs, ((L.M + 2 * pair::BM - 1) / (2 * pair::BM)) * (L.N / pair::BN));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = 2;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(pair::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = pair::SMEM_BYTES;
  cfg.stream = L.stream;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  CUtensorMap sA, sB, sR, sW;
  const int sf_rows = L.mx ? pair::SF_BOX_ROWS / 2 : pair::SF_BOX_ROWS;
  if (!make_sf_map(&sA, L.a_sf, ext.a, sf_rows) || !make_sf_map(&sB, L.b_sf, ext.b, sf_rows))
    return fail(QUADS_ERR_CUDA, "gemm: cuTensorMapEncodeTiled failed for the scale atoms");
  if (comp) {
    if (!make_sf_map(&sR, L.r_sf, ext.r, pair::SF_BOX_ROWS) ||
        !make_sf_map(&sW, ws_sf, ext.w, pair::SF_BOX_ROWS))
      return fail(QUADS_ERR_CUDA, "gemm: cuTensorMapEncodeTiled failed for the correction scales");
  } else {
    sR = sA;
    sW = sB;
  }
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, pair::pair_gemm_kernel, tA, tB, tR, tW, sA, sB, sR, sW, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(QUADS_ERR_CUDA, "gemm: launch of the CTA-pair kernel: %s", cudaGetErrorString(e));
  }
  return check_launch("gemm", launches);
}

void gemm_wait_test(int enable) { g_wait_test.store(enable ? 1 : 0); }
void gemm_timeline(unsigned long long* buf) { g_trace.store(buf); }
}  // namespace gemm

int read_gemm_device_error() {
  int v = 0;
  cudaMemcpyFromSymbol(&v, gemm::g_gemm_error, sizeof(int));
  int zero = 0;
  cudaMemcpyToSymbol(gemm::g_gemm_error, &zero, sizeof(int));
  return v;
}

int debug_line_gemm(long long* value) { return take_debug_line(value); }

}  // namespace quads

using namespace quads;

static bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Compensation operands: R_sel and sel, and either a prebuilt Q(W_sel) or the
// column-major weight copy it is built from.
static quads_status_t check_wsel_args(const char* who, const uint8_t* r_codes,
                                      const uint8_t* r_scales, const float* r_tensor_scale,
                                      const int32_t* sel, const uint8_t* w_codes_t,
                                      const uint8_t* w_scales_t, const uint8_t* w_sel_codes,
                                      const uint8_t* w_sel_scales, int32_t k, int64_t K) {
  if (!r_codes) return QUADS_OK;
  if (!r_scales || !r_tensor_scale || !sel || k <= 0 || k % 16 || k > K)
    return fail(QUADS_ERR_INVALID_ARG, "%s: compensation needs r_scales, r_tensor_scale, sel and 16<=k<=K, k%%16==0", who);
  if (!w_sel_codes != !w_sel_scales)
    return fail(QUADS_ERR_INVALID_ARG, "%s: give both w_sel_codes and w_sel_scales, or neither", who);
  if (w_sel_codes && (!al16(w_sel_codes) || !al16(w_sel_scales)))
    return fail(QUADS_ERR_MISALIGNED, "%s: Q(W_sel) must be 16-byte aligned", who);
  if (!w_sel_codes && (!w_codes_t || !w_scales_t))
    return fail(QUADS_ERR_INVALID_ARG, "%s: without a prebuilt Q(W_sel), compensation needs the column-major weight copy", who);
  return QUADS_OK;
}

extern "C" quads_status_t quads_w4a4_gemm_comp(int64_t M, int64_t N, int64_t K,
                                               const uint8_t* a_codes, const uint8_t* a_scales,
                                               const float* a_tensor_scale, const uint8_t* w_codes,
                                               const uint8_t* w_scales, const float* w_tensor_scale,
                                               const uint8_t* w_codes_t, const uint8_t* w_scales_t,
                                               const uint8_t* w_sel_codes,
                                               const uint8_t* w_sel_scales,
                                               const uint8_t* r_codes, const uint8_t* r_scales,
                                               const float* r_tensor_scale, const int32_t* sel,
                                               int32_t k, void* y, int32_t y_dtype, int64_t ldy,
                                               void* workspace, size_t workspace_bytes,
                                               void* stream) {
  if (M < 0 || N % 128 || N <= 0 || K % 64 || K <= 0)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "gemm: need M>=0, N%%128==0, K%%64==0 (M=%lld N=%lld K=%lld)", (long long)M, (long long)N, (long long)K);
  if (M == 0) return QUADS_OK;
  if (!a_codes || !a_scales || !a_tensor_scale || !w_codes || !w_scales || !w_tensor_scale || !y)
    return fail(QUADS_ERR_INVALID_ARG, "gemm: null operand pointer");
  if (M > (1ll << 31) - 256 || (int64_t)N * K / 2 > (1ll << 40))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "gemm: shape too large");
  if (y_dtype != QUADS_OUT_F32 && y_dtype != QUADS_OUT_BF16)
    return fail(QUADS_ERR_INVALID_ARG, "gemm: y_dtype");
  if (ldy < N || (y_dtype == QUADS_OUT_F32 ? ldy % 4 : ldy % 8))
    return fail(QUADS_ERR_MISALIGNED, "gemm: ldy must be >= N and keep 16-byte rows");
  if (!al16(a_codes) || !al16(w_codes) || !al16(a_scales) || !al16(w_scales) || !al16(y) ||
      (r_codes && (!al16(r_codes) || !al16(r_scales))))
    return fail(QUADS_ERR_MISALIGNED, "gemm: operands must be 16-byte aligned");
  if (quads_status_t st = check_wsel_args("gemm", r_codes, r_scales, r_tensor_scale, sel,
                                          w_codes_t, w_scales_t, w_sel_codes, w_sel_scales, k, K))
    return st;
  gemm::Launch L{};
  L.M = M; L.rows_cap = M; L.E = 1; L.N = (int)N; L.K = (int)K; L.k = k;
  L.kpad = r_codes ? quads_kpad(k) : 0;
  L.row_off = nullptr; L.row_cnt = nullptr;
  L.a = a_codes; L.a_sf = a_scales; L.b = w_codes; L.b_sf = w_scales;
  L.b_t = w_codes_t; L.b_sf_t = w_scales_t;
  L.wsel = w_sel_codes; L.wsel_sf = w_sel_scales;
  L.r = r_codes; L.r_sf = r_scales;
  L.a_ts = a_tensor_scale; L.b_ts = w_tensor_scale; L.r_ts = r_tensor_scale;
  L.a_pe = 0; L.r_pe = 0; L.sel = sel; L.sel_pe = 0;
  L.y = y; L.ldy = ldy; L.out_mode = y_dtype == QUADS_OUT_F32 ? gemm::OUT_F32 : gemm::OUT_BF16;
  L.y_amax = nullptr;
  L.ws = workspace; L.ws_bytes = workspace_bytes; L.stream = (cudaStream_t)stream;
  return gemm::launch(L);
}

extern "C" quads_status_t quads_moe_grouped_gemm(
    int32_t num_experts, int64_t rows_capacity, int64_t N, int64_t K,
    const int32_t* expert_offsets, const int32_t* expert_counts, const uint8_t* a_codes,
    const uint8_t* a_scales, const float* a_tensor_scale, int32_t a_scale_per_expert,
    const uint8_t* w_codes, const uint8_t* w_scales, const float* w_tensor_scale,
    const uint8_t* w_codes_t, const uint8_t* w_scales_t, const uint8_t* w_sel_codes,
    const uint8_t* w_sel_scales, const uint8_t* r_codes, const uint8_t* r_scales,
    const float* r_tensor_scale, int32_t r_scale_per_expert, const int32_t* sel, int32_t sel_per_expert, int32_t k,
    int32_t epilogue, void* y, int32_t y_dtype, int64_t ldy, float* y_amax, void* workspace,
    size_t workspace_bytes, void* stream) {
  if (!expert_offsets || !a_codes || !a_scales || !a_tensor_scale || !w_codes || !w_scales ||
      !w_tensor_scale || !y)
    return fail(QUADS_ERR_INVALID_ARG, "moe_gemm: null operand pointer");
  if (num_experts < 1 || num_experts > gemm::MAX_GROUPS || rows_capacity < 1 ||
      rows_capacity % 128 || N % 128 || N <= 0 ||
      K % 64 || K <= 0)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "moe_gemm: need experts>=1, rows_capacity%%128==0, N%%128==0, K%%64==0");
  if (epilogue != QUADS_EPILOGUE_NONE && epilogue != QUADS_EPILOGUE_SWIGLU)
    return fail(QUADS_ERR_INVALID_ARG, "moe_gemm: epilogue");
  if (epilogue == QUADS_EPILOGUE_SWIGLU && y_dtype != QUADS_OUT_BF16)
    return fail(QUADS_ERR_INVALID_ARG, "moe_gemm: SWIGLU writes bf16");
  const int64_t ycols = epilogue == QUADS_EPILOGUE_SWIGLU ? N / 2 : N;
  if (ldy < ycols || (y_dtype == QUADS_OUT_F32 ? ldy % 4 : ldy % 8))
    return fail(QUADS_ERR_MISALIGNED, "moe_gemm: ldy");
  if (!al16(a_codes) || !al16(w_codes) || !al16(a_scales) || !al16(w_scales) || !al16(y) ||
      (r_codes && (!al16(r_codes) || !al16(r_scales))))
    return fail(QUADS_ERR_MISALIGNED, "moe_gemm: operands must be 16-byte aligned");
  if (quads_status_t st = check_wsel_args("moe_gemm", r_codes, r_scales, r_tensor_scale, sel,
                                          w_codes_t, w_scales_t, w_sel_codes, w_sel_scales, k, K))
    return st;
  gemm::Launch L{};
  L.M = rows_capacity; L.rows_cap = rows_capacity; L.E = num_experts; L.N = (int)N; L.K = (int)K;
  L.k = k; L.kpad = r_codes ? quads_kpad(k) : 0;
  L.row_off = expert_offsets; L.row_cnt = expert_counts;
  L.a = a_codes; L.a_sf = a_scales; L.b = w_codes; L.b_sf = w_scales;
  L.b_t = w_codes_t; L.b_sf_t = w_scales_t;
  L.wsel = w_sel_codes; L.wsel_sf = w_sel_scales;
  L.r = r_codes; L.r_sf = r_scales;
  L.a_ts = a_tensor_scale; L.b_ts = w_tensor_scale; L.r_ts = r_tensor_scale;
  L.a_pe = a_scale_per_expert; L.r_pe = r_scale_per_expert; L.sel = sel; L.sel_pe = sel_per_expert;
  L.y = y; L.ldy = ldy; L.y_amax = y_amax;
  L.out_mode = epilogue == QUADS_EPILOGUE_SWIGLU ? gemm::OUT_SWIGLU
               : (y_dtype == QUADS_OUT_F32 ? gemm::OUT_F32 : gemm::OUT_BF16);
  L.ws = workspace; L.ws_bytes = workspace_bytes; L.stream = (cudaStream_t)stream;
  return gemm::launch(L);
}

extern "C" quads_status_t quads_mx_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* a_codes,
                                        const uint8_t* a_scales, const uint8_t* w_codes,
                                        const uint8_t* w_scales, void* y, int32_t y_dtype,
                                        int64_t ldy, void* stream) {
  if (M < 0 || N % 128 || N <= 0 || K % 128 || K <= 0)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "mx_gemm: need M>=0, N%%128==0, K%%128==0 (M=%lld N=%lld K=%lld)", (long long)M, (long long)N, (long long)K);
  if (M == 0) return QUADS_OK;
  if (!a_codes || !a_scales || !w_codes || !w_scales || !y)
    return fail(QUADS_ERR_INVALID_ARG, "mx_gemm: null operand pointer");
  if (M > (1ll << 31) - 256 || (int64_t)N * K / 2 > (1ll << 40))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "mx_gemm: shape too large");
  if (y_dtype != QUADS_OUT_F32 && y_dtype != QUADS_OUT_BF16)
    return fail(QUADS_ERR_INVALID_ARG, "mx_gemm: y_dtype");
  if (ldy < N || (y_dtype == QUADS_OUT_F32 ? ldy % 4 : ldy % 8))
    return fail(QUADS_ERR_MISALIGNED, "mx_gemm: ldy must be >= N and keep 16-byte rows");
  if (!al16(a_codes) || !al16(w_codes) || !al16(a_scales) || !al16(w_scales) || !al16(y))
    return fail(QUADS_ERR_MISALIGNED, "mx_gemm: operands must be 16-byte aligned");
  gemm::Launch L{};
  L.M = M; L.rows_cap = M; L.E = 1; L.N = (int)N; L.K = (int)K; L.k = 0; L.kpad = 0;
  L.row_off = nullptr; L.row_cnt = nullptr;
  L.a = a_codes; L.a_sf = a_scales; L.b = w_codes; L.b_sf = w_scales;
  L.a_ts = nullptr; L.b_ts = nullptr; L.r_ts = nullptr;
  L.a_pe = 0; L.r_pe = 0; L.sel = nullptr; L.sel_pe = 0;
  L.y = y; L.ldy = ldy; L.out_mode = y_dtype == QUADS_OUT_F32 ? gemm::OUT_F32 : gemm::OUT_BF16;
  L.mx = 1;
  L.y_amax = nullptr;
  L.stream = (cudaStream_t)stream;
  return gemm::launch(L);
}

extern "C" void quads_test_gemm_wait_timeout(int32_t enable) { gemm::gemm_wait_test(enable); }

extern "C" int32_t quads_set_gemm_tile_policy(int32_t policy) {
  if (policy != QUADS_GEMM_TILES_AUTO && policy != QUADS_GEMM_TILES_128 &&
      policy != QUADS_GEMM_TILES_256)
    return -1;
  return gemm::g_tile_policy.exchange(policy);
}

extern "C" void quads_test_gemm_timeline(uint64_t* device_buffer) {
  gemm::gemm_timeline(reinterpret_cast<unsigned long long*>(device_buffer));
}

extern "C" quads_status_t quads_weight_columns(const uint8_t* w_codes, const uint8_t* w_scales,
                                               int32_t num_groups, int64_t rows_per_group,
                                               int64_t cols, uint8_t* codes_t, uint8_t* scales_t,
                                               void* stream) {
  if (!w_codes || !w_scales || !codes_t || !scales_t)
    return fail(QUADS_ERR_INVALID_ARG, "weight_columns: null pointer argument");
  if (num_groups < 1 || rows_per_group <= 0 || rows_per_group % 128 || cols <= 0 || cols % 64)
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "weight_columns: rows_per_group %% 128 and cols %% 64");
  const int64_t blocks = (int64_t)num_groups * (rows_per_group / 128) * (cols / 64);
  if (blocks >= ((int64_t)1 << 31))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "weight_columns: too many 128x64 blocks");
  gemm::wtrans_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      w_codes, w_scales, num_groups, (int)rows_per_group, (int)cols, codes_t, scales_t);
  return check_launch("weight_columns", 1);
}

extern "C" quads_status_t quads_select_weight_channels(
    int32_t num_groups, int64_t rows_per_group, int64_t cols, const uint8_t* codes_t,
    const uint8_t* scales_t, const int32_t* sel, int32_t sel_per_group, int32_t k,
    uint8_t* w_sel_codes, uint8_t* w_sel_scales, void* stream) {
  if (!codes_t || !scales_t || !sel || !w_sel_codes || !w_sel_scales)
    return fail(QUADS_ERR_INVALID_ARG, "select_weight_channels: null pointer argument");
  if (num_groups < 1 || num_groups > 65535 || rows_per_group <= 0 || rows_per_group % 128 ||
      rows_per_group > (1 << 30) || cols <= 0 || cols % 64 || cols > (1 << 30))
    return fail(QUADS_ERR_UNSUPPORTED_SHAPE, "select_weight_channels: rows_per_group %% 128, cols %% 64, groups <= 65535");
  if (k <= 0 || k % 16 || k > cols)
    return fail(QUADS_ERR_INVALID_ARG, "select_weight_channels: need 16 <= k <= cols, k %% 16 == 0");
  if (!al16(w_sel_codes) || !al16(w_sel_scales) || !al16(codes_t) || !al16(scales_t))
    return fail(QUADS_ERR_MISALIGNED, "select_weight_channels: codes_t, scales_t, w_sel_codes and w_sel_scales must be 16-byte aligned");
  const int kpad = quads_kpad(k);
  gemm::launch_wsel(codes_t, scales_t, num_groups, (int)rows_per_group, (int)cols, sel,
                    sel_per_group, k, kpad, w_sel_codes, w_sel_scales, (cudaStream_t)stream);
  return check_launch("select_weight_channels", 1);
}
