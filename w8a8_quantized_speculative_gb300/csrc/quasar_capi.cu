// Library-wide C-ABI pieces: status strings, version, the device error word
// and the wait limit used by every bounded device-side wait.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "quasar_common.cuh"

namespace quasar {

// Site code of the first device-side wait that ran out since the last
// quasar_get_device_error() (0 = none).  One word per device image.
__device__ unsigned int g_error_word = 0;

namespace {
constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
unsigned int* g_err_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
std::mutex g_mu;
}  // namespace

unsigned int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = reinterpret_cast<unsigned int*>(p);
  }
  return g_err_ptr[dev];
}

unsigned long long wait_limit_ns() { return g_wait_ns.load(); }

// Self-test of the bounded waits: one thread waits on an mbarrier that
// nothing ever completes, runs out after limit_ns, records SITE_SELFTEST and
// returns.
__global__ void wait_selftest_kernel(unsigned int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, &abort_flag, err, SITE_SELFTEST, limit_ns);
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

// The driver's tensor-map encoder, resolved through the runtime so that the
// library needs no link-time dependency on libcuda.
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool encode_2d_u8(CUtensorMap* map, const void* base, int inner, int outer, int box_inner, int box_outer) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)inner};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_2d_bf16(CUtensorMap* map, const void* base, int inner, int outer, long long ld, int box_inner,
                    int box_outer) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

quasar_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? QUASAR_OK : QUASAR_ERR_CUDA; }

}  // namespace quasar

extern "C" {

const char* quasar_status_string(int status) {
  switch (status) {
    case QUASAR_OK: return "ok";
    case QUASAR_ERR_INVALID_ARG: return "invalid argument";
    case QUASAR_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case QUASAR_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case QUASAR_ERR_CUDA: return "CUDA runtime/driver error";
    case QUASAR_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int quasar_version(void) { return (1 << 16) | 0; }

quasar_status_t quasar_set_wait_limit_ns(uint64_t ns) {
  quasar::g_wait_ns.store(ns ? ns : quasar::kDefaultWaitNs);
  return QUASAR_OK;
}

quasar_status_t quasar_selftest_wait_timeout(uint64_t limit_ns, quasar_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000ull) return QUASAR_ERR_INVALID_ARG;
  unsigned int* err = quasar::device_error_word();
  if (!err) return QUASAR_ERR_CUDA;
  quasar::wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, limit_ns);
  return quasar::cuda_status(cudaGetLastError());
}

quasar_status_t quasar_get_device_error(quasar_stream_t stream, uint32_t* site) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return QUASAR_ERR_CUDA;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, quasar::g_error_word, sizeof(v));
  if (e != cudaSuccess) return QUASAR_ERR_CUDA;
  if (site) *site = v;
  if (v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(quasar::g_error_word, &zero, sizeof(zero)) != cudaSuccess) return QUASAR_ERR_CUDA;
    return QUASAR_ERR_TIMEOUT;
  }
  return QUASAR_OK;
}

}  // extern "C"
