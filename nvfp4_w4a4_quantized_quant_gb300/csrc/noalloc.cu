// Residual-channel selection for callers that cannot allocate device memory.
//
// quads_select_residual_channels needs scratch (the float32 residual slice, its
// per-group maxima and the per-group channel scores) that its caller passes in
// as `workspace`.  Some callers have no way to provide it: a host runtime that
// hands out only the tensors it owns (inputs and outputs) and forbids
// allocation while it runs, a CUDA-graph-capturing framework whose memory pool
// is frozen for the capture, or an embedding process that never links an
// allocator.  quads_select_residual_channels_noalloc serves them with a fixed
// scratch array compiled into the library instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  Host code cannot use the array's
// name as a device address; its device address is looked up once per device
// with cudaGetSymbolAddress (on the first call on that device, with the device
// current) and cached.
#include <mutex>

#include "common.cuh"

namespace quads {

static __device__ __align__(256) unsigned char g_select_scratch[QUADS_NOALLOC_SELECT_SCRATCH_BYTES];

static void* scratch_address(int device, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[128] = {nullptr};
  *err = cudaSuccess;
  if (device < 0 || device >= 128) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    addr[device] = p;
  }
  return addr[device];
}

}  // namespace quads

using namespace quads;

extern "C" quads_status_t quads_select_residual_channels_noalloc(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* group_offsets,
    int32_t num_groups, const int32_t* group_counts, const uint8_t* scales, int32_t scale_layout,
    const float* tensor_scale, const float* score_partials, int32_t k, int32_t* sel,
    float* scores_out, uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout,
    float* r_tensor_scale, void* stream) {
  // the same argument checks, in the same order, as the workspace entry point
  size_t need = 0;
  if (quads_status_t s = select_check_args(x, rows, cols, ldx, group_offsets, num_groups,
                                           group_counts, scales, tensor_scale, score_partials, k,
                                           sel, r_codes, r_scales, r_tensor_scale, &need))
    return s;
  if (rows > 0 && need > (size_t)QUADS_NOALLOC_SELECT_SCRATCH_BYTES)
    return fail(QUADS_ERR_WORKSPACE,
                "select_noalloc: this shape needs %zu bytes of scratch, the built-in array holds %zu "
                "(rows*k*4 + per-group maxima + groups*cols*4 must fit)",
                need, (size_t)QUADS_NOALLOC_SELECT_SCRATCH_BYTES);
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return fail(QUADS_ERR_CUDA, "select_noalloc: %s", cudaGetErrorString(e));
  void* scratch = scratch_address(device, &e);
  if (!scratch)
    return fail(QUADS_ERR_CUDA, "select_noalloc: cudaGetSymbolAddress failed: %s",
                cudaGetErrorString(e));
  return quads_select_residual_channels(x, rows, cols, ldx, group_offsets, num_groups,
                                        group_counts, scales, scale_layout, tensor_scale,
                                        score_partials, k, sel,
                                        scores_out, r_codes, r_scales, r_scale_layout,
                                        r_tensor_scale, scratch,
                                        (size_t)QUADS_NOALLOC_SELECT_SCRATCH_BYTES, nullptr,
                                        stream);
}
