// A0: offline calibration of the smoothing vector.
//
// Quasar summary zh §2 "方法论": the smoothing factor s is calibrated offline
// and the identity Y = (W·diag(s)^-1)·(diag(s)·X) moves quantization
// difficulty from the activations to the weights.  Here s multiplies X, so
//   smooth[k] = max_n|W[n][k]|^(1-alpha) / max_m|Xcal[m][k]|^alpha
// (SmoothQuant's migration factor inverted), with smooth[k] = 1 when either
// maximum is 0.  Column maxima are exact (BF16 magnitudes compared as
// integers); the ratio is formed in fp64 -- for alpha = 0.5 with IEEE sqrt and
// division, so it is correctly rounded -- and rounded once to fp32.
#include "quasar_common.cuh"

namespace quasar {
namespace calib {

constexpr int THREADS = 128;
constexpr int ROWS_PER_BLOCK = 64;

// Column-wise max |value| of a BF16 matrix, as fp32 bit patterns (non-negative
// floats order like their bit patterns), merged with atomicMax into out[K].
__global__ void colmax_kernel(const uint16_t* __restrict__ in, int rows, int ld, int K, unsigned int* out) {
  const int v = blockIdx.x * THREADS + threadIdx.x;  // 8-column group
  if (v * 8 >= K) return;
  const int r0 = blockIdx.y * ROWS_PER_BLOCK;
  const int r1 = min(rows, r0 + ROWS_PER_BLOCK);
  uint32_t m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int r = r0; r < r1; ++r) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(in + (size_t)r * ld) + v);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[2 * i] = max(m[2 * i], w[i] & 0x7FFFu);
      m[2 * i + 1] = max(m[2 * i + 1], (w[i] >> 16) & 0x7FFFu);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (m[i]) atomicMax(&out[v * 8 + i], m[i] << 16);
}

__global__ void finalize_kernel(const unsigned int* __restrict__ xmax, const unsigned int* __restrict__ wmax, int K,
                                float alpha, float* __restrict__ smooth) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= K) return;
  const double xm = (double)__uint_as_float(xmax[k]);
  const double wm = (double)__uint_as_float(wmax[k]);
  double s = 1.0;
  if (xm > 0.0 && wm > 0.0) {
    if (alpha == 0.5f)
      s = sqrt(wm) / sqrt(xm);
    else
      s = pow(wm, 1.0 - (double)alpha) / pow(xm, (double)alpha);
  }
  smooth[k] = __double2float_rn(s);
}

}  // namespace calib
}  // namespace quasar

extern "C" {

size_t quasar_calibrate_workspace_size(int K) { return K > 0 ? (size_t)2 * K * sizeof(unsigned int) : 0; }

quasar_status_t quasar_calibrate_smooth(const void* Xcal_bf16, int Mcal, int ldx, const void* W_bf16, int N,
                                        int ldw, int K, float alpha, float* smooth, void* workspace,
                                        size_t ws_bytes, quasar_stream_t stream_) {
  using namespace quasar;
  if (!Xcal_bf16 || !W_bf16 || !smooth || Mcal <= 0 || N <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (!(alpha > 0.f && alpha < 1.f)) return QUASAR_ERR_INVALID_ARG;
  if (K % 8 != 0 || ldx < K || ldw < K || ldx % 8 != 0 || ldw % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (!aligned(Xcal_bf16, 16) || !aligned(W_bf16, 16) || !aligned(smooth, 4)) return QUASAR_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < quasar_calibrate_workspace_size(K) || !aligned(workspace, 4))
    return QUASAR_ERR_WORKSPACE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  unsigned int* xmax = reinterpret_cast<unsigned int*>(workspace);
  unsigned int* wmax = xmax + K;
  cudaError_t e = cudaMemsetAsync(workspace, 0, (size_t)2 * K * sizeof(unsigned int), stream);
  if (e != cudaSuccess) return cuda_status(e);
  const int gx = (K / 8 + calib::THREADS - 1) / calib::THREADS;
  calib::colmax_kernel<<<dim3(gx, (Mcal + calib::ROWS_PER_BLOCK - 1) / calib::ROWS_PER_BLOCK), calib::THREADS, 0,
                         stream>>>(reinterpret_cast<const uint16_t*>(Xcal_bf16), Mcal, ldx, K, xmax);
  calib::colmax_kernel<<<dim3(gx, (N + calib::ROWS_PER_BLOCK - 1) / calib::ROWS_PER_BLOCK), calib::THREADS, 0,
                         stream>>>(reinterpret_cast<const uint16_t*>(W_bf16), N, ldw, K, wmax);
  calib::finalize_kernel<<<(K + 255) / 256, 256, 0, stream>>>(xmax, wmax, K, alpha, smooth);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
