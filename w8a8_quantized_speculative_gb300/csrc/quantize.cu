// A1 (offline weight packing) and A2 (online activation smooth + quantize).
//
// Quasar summary pt §2 "Metodologia" steps 1-2, zh §2 "方法论": weights are
// smoothed (divided by s) and quantized to INT8 offline; during verification
// the BF16 activations are smoothed (multiplied by s) and quantized on the
// fly.  Both are the same per-row symmetric quantizer:
//   v[k]  = float(in[k]) op smooth[k]        (op = * for activations, / for weights)
//   a     = max_k |v[k]|
//   scale = a / 127                          (0 if a == 0)
//   q[k]  = clamp(rne(v[k] * (127 / a)), -127, 127)
// in fp32 with IEEE rounding (division and multiply correctly rounded, no
// contraction).  One CTA per row: 128-bit loads of 8 BF16 values, warp-shuffle
// absmax, then a second pass that re-derives v (bit-identical) and stores
// 8 codes per 64-bit store.  Rows are short (<= 24 KB) and the second pass
// is served from L1/L2.
#include <algorithm>

#include "quasar_common.cuh"

namespace quasar {
namespace quant {

constexpr int THREADS = 256;

template <bool DIVIDE>
QUASAR_DEVICE_INLINE float smooth_op(float x, float s) {
  return DIVIDE ? __fdiv_rn(x, s) : __fmul_rn(x, s);
}

QUASAR_DEVICE_INLINE void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <bool DIVIDE>
__global__ void __launch_bounds__(THREADS) quant_rows_kernel(const uint16_t* __restrict__ in, int ld,
                                                             const float* __restrict__ smooth, int K,
                                                             int8_t* __restrict__ q, float* __restrict__ scale) {
  const int row = blockIdx.x;
  const uint16_t* src = in + (size_t)row * ld;
  const int nvec = K / 8;

  // Pass 1: absmax of the smoothed row.
  float amax = 0.f;
  for (int v = threadIdx.x; v < nvec; v += THREADS) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src) + v);
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v);
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v + 1);
    float f[8];
    bf16x8_to_f32(raw, f);
    const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(smooth_op<DIVIDE>(f[i], s[i])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[THREADS / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float a = threadIdx.x < THREADS / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (threadIdx.x == 0) red[0] = a;
  }
  __syncthreads();
  amax = red[0];

  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;

  // Pass 2: codes.
  int8_t* dst = q + (size_t)row * K;
  for (int v = threadIdx.x; v < nvec; v += THREADS) {
    uint32_t packed[2] = {0u, 0u};
    if (amax > 0.f) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src) + v);
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v);
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v + 1);
      float f[8];
      bf16x8_to_f32(raw, f);
      const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int c = __float2int_rn(__fmul_rn(smooth_op<DIVIDE>(f[i], s[i]), inv));
        c = max(-127, min(127, c));
        packed[i >> 2] |= (uint32_t)(c & 0xFF) << (8 * (i & 3));
      }
    }
    reinterpret_cast<uint2*>(dst)[v] = make_uint2(packed[0], packed[1]);
  }
}

template <bool DIVIDE>
static quasar_status_t run(const void* in, int ld, const float* smooth, int rows, int K, int8_t* q, float* scale,
                           cudaStream_t stream) {
  if (rows < 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || ld < K || ld % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (rows == 0) return QUASAR_OK;  // empty batch: nothing is read or written
  if (!in || !smooth || !q || !scale) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(in, 16) || !aligned(smooth, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return QUASAR_ERR_UNSUPPORTED;
  quant_rows_kernel<DIVIDE><<<rows, THREADS, 0, stream>>>(reinterpret_cast<const uint16_t*>(in), ld, smooth, K,
                                                          q, scale);
  return cuda_status(cudaGetLastError());
}

}  // namespace quant
}  // namespace quasar

extern "C" {

quasar_status_t quasar_pack_weights(const void* W_bf16, int ldw, const float* smooth, int N, int K, int8_t* Wq,
                                    float* sw, quasar_stream_t stream) {
  if (N <= 0) return QUASAR_ERR_INVALID_ARG;
  return quasar::quant::run<true>(W_bf16, ldw, smooth, N, K, Wq, sw, reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_smooth_quant_act(const void* X_bf16, int ldx, const float* smooth, int M, int K,
                                        int8_t* Xq, float* sa, quasar_stream_t stream) {
  return quasar::quant::run<false>(X_bf16, ldx, smooth, M, K, Xq, sa, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
