// Host-side glue of the libquads C ABI: status strings, per-thread error
// detail, workspace sizing and the device error word.
#include <atomic>
#include <cstdarg>
#include <cstdio>

#include "common.cuh"

namespace quads {

static thread_local char g_detail[512] = "";

void set_detail(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
}

quads_status_t fail(quads_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return s;
}

static std::atomic<unsigned long long> g_launches{0};

quads_status_t check_launch(const char* what, int kernels_launched) {
  g_launches += (unsigned long long)kernels_launched;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(QUADS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return QUADS_OK;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

int read_quant_device_error(cudaStream_t);
int read_gemm_device_error();
int debug_line_quantize(long long* value);
int debug_line_gemm(long long* value);
int debug_line_moe(long long* value);

}  // namespace quads

using namespace quads;

extern "C" int quads_version(void) { return 100; }

extern "C" uint64_t quads_kernel_launch_count(void) { return (uint64_t)g_launches.load(); }

extern "C" const char* quads_status_string(quads_status_t s) {
  switch (s) {
    case QUADS_OK: return "ok";
    case QUADS_ERR_INVALID_ARG: return "invalid argument";
    case QUADS_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case QUADS_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
    case QUADS_ERR_CUDA: return "CUDA error";
    case QUADS_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case QUADS_ERR_DEVICE_CHECK: return "device-side argument check failed";
    case QUADS_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

extern "C" const char* quads_last_error_detail(void) { return g_detail; }

extern "C" int32_t quads_kpad(int32_t k) {
  if (k <= 64) return 64;
  if (k <= 128) return 128;
  if (k <= 256) return 256;
  return (k + 255) / 256 * 256;
}

extern "C" size_t quads_workspace_size(int32_t op, int64_t rows, int64_t cols, int64_t n,
                                       int32_t k, int32_t num_groups) {
  const size_t G = num_groups > 0 ? (size_t)num_groups : 1;
  switch (op) {
    case QUADS_OP_QUANTIZE:
      return G * 4;
    case QUADS_OP_SELECT:  // residual slice, per-group amax, per-group channel scores
      return (((size_t)rows * (size_t)k * 4 + 255) & ~(size_t)255) + ((G * 4 + 255) & ~(size_t)255) +
             G * (size_t)cols * 4;
    case QUADS_OP_QUANTIZE_SELECT: {  // control words, partials, scores, residual slice
      const size_t r = rows > 0 ? (size_t)rows : 0, c = cols > 0 ? (size_t)cols : 0;
      const size_t kk = k > 0 ? (size_t)k : 0;
      auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
      return 256 + al((r + 31) / 32 * c * 4) + al(c * 4) + al(r * kk * 4);
    }
    case QUADS_OP_QUANTIZE_SELECT_GROUPS:  // residual slice
      return rows > 0 && k > 0 ? (size_t)rows * (size_t)k * 4 : 0;
    case QUADS_OP_MOE_ROUTE:  // per-32-token-block expert counts and prefixes: rows = tokens, cols = experts
      return (size_t)((rows > 0 ? rows : 0) + 31) / 32 * (size_t)(cols > 0 ? cols : 0) * 8 + 16;
    case QUADS_OP_GEMM:
    case QUADS_OP_MOE_GEMM: {
      const size_t e = op == QUADS_OP_MOE_GEMM ? G : 1;
      const size_t kp = (size_t)quads_kpad(k);
      const size_t brows = e * (size_t)n;
      return ((brows * kp / 2 + 1023) & ~(size_t)1023) + brows * kp / 16;
    }
  }
  (void)cols;
  return 0;
}

extern "C" quads_status_t quads_device_status(void* stream, int32_t* device_code) {
  if (!device_code) return fail(QUADS_ERR_INVALID_ARG, "device_status: null output");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(QUADS_ERR_CUDA, "device_status: %s", cudaGetErrorString(e));
  int g = read_gemm_device_error();
  int q = read_quant_device_error((cudaStream_t)stream);
  *device_code = g ? g : q;
  // bounds-checked builds: the first failed guard of each source file
  long long vq = 0, vg = 0, vm = 0;
  const int lq = debug_line_quantize(&vq), lg = debug_line_gemm(&vg), lm = debug_line_moe(&vm);
  if (lq || lg || lm) {
    *device_code = QUADS_ERR_DEVICE_CHECK;
    set_detail("bounds check failed: quantize.cu:%d (%lld) gemm.cu:%d (%lld) moe.cu:%d (%lld) "
               "(line 0 = none; the value recorded with the first failure)",
               lq, vq, lg, vg, lm, vm);
  }
  return QUADS_OK;
}
