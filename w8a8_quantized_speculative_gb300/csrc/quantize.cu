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
// absmax, then a second pass that stores 8 codes per 64-bit store.  Activation
// rows of up to 12288 values keep the whole row in registers (one memory
// round trip); longer rows and the weights re-derive v in the second pass
// (bit-identical), served from L1/L2.
//
// The MLP block's glue before down takes the same activation path on
// h = bf16_rne(silu(gate) * up) computed from the gate_up output row as it is
// loaded (quasar_silu_mul_smooth_quant): the pages dequantize to BF16 ahead of
// the nonlinear layers, and down then re-smooths and re-quantizes.
//
// Activation codes are written row-major [M][K].  Weight codes are written in
// the packed layout the W8A8 linear streams: 128 x 128 blocks, tile-major,
// each block 16 KB contiguous with the 16-byte chunks of row r stored in
// 128B-swizzled order (chunk c at position c ^ (r % 8)), each byte holding
// code + 128; see quasar.h.
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

// The MLP glue before down (SiLU(gate) * up, rounded once to BF16) needs an
// exponential whose every bit is fixed, because the rounded h decides the
// codes.  exp_cw: Cody and Waite's argument reduction t = n ln2 + r, with
// ln2 split in a 15-bit head (n * head is exact for |n| < 2^9) and a tail,
// then the degree-7 Taylor polynomial of e^r by Horner, times 2^n.  Each step
// is one correctly rounded fp32 operation (no contraction); within 2 ulp of
// e^t on [-87, 88], the range callers clamp to (2^n stays a normal number).
QUASAR_DEVICE_INLINE float exp_cw(float t) {
  const float n = rintf(__fmul_rn(t, __uint_as_float(0x3FB8AA3Bu)));                   // t / ln2
  const float r = __fsub_rn(__fsub_rn(t, __fmul_rn(n, __uint_as_float(0x3F317200u))),  // ln2 head
                            __fmul_rn(n, __uint_as_float(0x35BFBE8Eu)));                // ln2 tail
  float p = __uint_as_float(0x39500D01u);                                                // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3AB60B61u));                         // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3C088889u));                         // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3D2AAAABu));                         // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3E2AAAABu));                         // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  return __fmul_rn(p, __uint_as_float((uint32_t)((int)n + 127) << 23));
}

// h = bf16_rne(silu(g) * u) as fp32, silu(g) = g / (1 + exp(-g)) with the
// exponential's argument clamped to [-87, 88].
QUASAR_DEVICE_INLINE float silu_mul_bf16(float g, float u) {
  const float t = fminf(fmaxf(-g, -87.f), 88.f);
  const float s = __fdiv_rn(g, __fadd_rn(1.f, exp_cw(t)));
  return __bfloat162float(__float2bfloat16_rn(__fmul_rn(s, u)));
}

// GLU rows hold [gate (K values) | up (K values)]: replace the 8 gate values
// in f by h = silu(gate) * up.
QUASAR_DEVICE_INLINE void glu8(float (&f)[8], const uint4& up) {
  float u[8];
  bf16x8_to_f32(up, u);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = silu_mul_bf16(f[i], u[i]);
}

// Byte offset of code (n, k) in the packed weight layout (k a multiple of 8).
QUASAR_DEVICE_INLINE size_t packed_offset(int n, int k, int KB) {
  const int r = n & 127, kk = k & 127, c = kk >> 4;
  return (((size_t)(n >> 7) * KB + (k >> 7)) * 128 + r) * 128 + ((c ^ (r & 7)) << 4) + (kk & 15);
}

template <bool DIVIDE, bool PACKED, bool GLU = false>
__global__ void __launch_bounds__(THREADS) quant_rows_kernel(const uint16_t* __restrict__ in, int ld,
                                                             const float* __restrict__ smooth, int K,
                                                             int8_t* __restrict__ q, float* __restrict__ scale) {
  // Launched with programmatic dependent launch: let the next kernel start
  // its independent prologue (e.g. a GEMM's weight stream) at once, then
  // wait until the previous kernel's writes (our input) are visible.
  pdl_launch_dependents();
  pdl_wait();
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
    if constexpr (GLU) glu8(f, __ldg(reinterpret_cast<const uint4*>(src + K) + v));
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
  const int KB = (K + 127) >> 7;
  for (int v = threadIdx.x; v < nvec; v += THREADS) {
    uint32_t packed[2] = {0u, 0u};
    if (amax > 0.f) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src) + v);
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v);
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v + 1);
      float f[8];
      bf16x8_to_f32(raw, f);
      if constexpr (GLU) glu8(f, __ldg(reinterpret_cast<const uint4*>(src + K) + v));
      const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int c = __float2int_rn(__fmul_rn(smooth_op<DIVIDE>(f[i], s[i]), inv));
        c = max(-127, min(127, c));
        packed[i >> 2] |= (uint32_t)(c & 0xFF) << (8 * (i & 3));
      }
    }
    if (PACKED)  // packed weight bytes hold code + 128
      *reinterpret_cast<uint2*>(q + packed_offset(row, 8 * v, KB)) =
          make_uint2(packed[0] ^ 0x80808080u, packed[1] ^ 0x80808080u);
    else
      reinterpret_cast<uint2*>(dst)[v] = make_uint2(packed[0], packed[1]);
  }
}

// Activation rows of up to THREADS * 8 * VPT values: every load of the row
// (and of its smoothing factors) is issued before any is used, both passes
// run from registers, so a row costs one memory round trip.  This matters
// on the verification path: the quantizer runs while the next linear's
// weight stream already fills the memory system, and each dependent round
// trip then waits behind it.  Same arithmetic as quant_rows_kernel<false,
// false>.
//
// `xh` (optional): the same codes as fp16 [rows][K] (exact), for a linear that
// takes its token operand already widened.  GLU: the row is [gate | up] and
// the values quantized are h = bf16_rne(silu(gate) * up).
template <int VPT, bool GLU = false>
__global__ void __launch_bounds__(THREADS) quant_act_kernel(const uint16_t* __restrict__ in, int ld,
                                                            const float* __restrict__ smooth, int K,
                                                            int8_t* __restrict__ q, float* __restrict__ scale,
                                                            uint4* __restrict__ xh) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const uint16_t* src = in + (size_t)row * ld;
  const int nvec = K / 8;
  uint4 raw[VPT];
  uint4 rawu[GLU ? VPT : 1];
  float4 sm[2 * VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v < nvec) {
      raw[i] = __ldg(reinterpret_cast<const uint4*>(src) + v);
      if constexpr (GLU) rawu[i] = __ldg(reinterpret_cast<const uint4*>(src + K) + v);
      sm[2 * i] = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v);
      sm[2 * i + 1] = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v + 1);
    }
  }
  float x[VPT][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    bf16x8_to_f32(raw[i], x[i]);
    if constexpr (GLU) {
      if (v < nvec) glu8(x[i], rawu[i]);
    }
    const float s[8] = {sm[2 * i].x, sm[2 * i].y, sm[2 * i].z, sm[2 * i].w,
                        sm[2 * i + 1].x, sm[2 * i + 1].y, sm[2 * i + 1].z, sm[2 * i + 1].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[i][e] = __fmul_rn(x[i][e], s[e]);
      if (v < nvec) amax = fmaxf(amax, fabsf(x[i][e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[THREADS / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
  int8_t* dst = q + (size_t)row * K;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v >= nvec) continue;
    uint32_t packed[2] = {0u, 0u};
    if (amax > 0.f) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int c = __float2int_rn(__fmul_rn(x[i][e], inv));
        c = max(-127, min(127, c));
        packed[e >> 2] |= (uint32_t)(c & 0xFF) << (8 * (e & 3));
      }
    }
    reinterpret_cast<uint2*>(dst)[v] = make_uint2(packed[0], packed[1]);
    if (xh) {
      uint4 h;
      s8x4_to_f16x4(packed[0], h.x, h.y);
      s8x4_to_f16x4(packed[1], h.z, h.w);
      xh[(size_t)row * nvec + v] = h;
    }
  }
}

QUASAR_DEVICE_INLINE float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// RMSNorm ahead of a linear (qkv, gate_up) fused with its smooth + quantize,
// one CTA per row of up to 2048 VPT values, every load issued up front as in
// quant_act_kernel.  Per row: ss = sum of the squares of the BF16 inputs.  A
// BF16 value has 8 significant bits, so its square is exact in fp32 (inside
// [2^-120, 2^120]); each thread sums each group of eight squares in fp32 with
// Neumaier's compensation (every rounding error of the running sum is
// recovered exactly and kept in a second term) and adds the two terms of
// each group to an fp64 total; a thread holding a value outside [2^-60,
// 2^60] (where a square could leave fp32's normal range) sums its squares in
// fp64 instead.  The thread totals are added in fp64 (a butterfly across the
// warp, the warps in order); r = fp32_rn(1 / sqrt(ss / K + eps)) with IEEE
// fp64 division and square root; t = bf16(x * r), h = bf16(t * gamma); then
// the A2 quantizer on fp32(h) * smooth.  The per-group compensation errors
// (below 64 x 2^-48 of the group's sum) and the order of the fp64 additions
// move ss by well under 2^-39 relative from the correctly rounded sum, which
// changes r only when 1 / sqrt(...) lies within a hair (2^-38 relative) of an
// fp32 rounding midpoint.  (GB300 issues fp64 at a small fraction of the fp32
// rate: an all-fp64 sum took ~15 us for 288 rows of 4096.)
template <int VPT>
__global__ void __launch_bounds__(THREADS) rms_quant_kernel(const uint16_t* __restrict__ in, int ld,
                                                            const uint16_t* __restrict__ gamma, float eps,
                                                            const float* __restrict__ smooth, int K,
                                                            int8_t* __restrict__ q, float* __restrict__ scale) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const uint16_t* src = in + (size_t)row * ld;
  const int nvec = K / 8;
  uint4 raw[VPT], gw[VPT];
  float4 sm[2 * VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v < nvec) {
      raw[i] = __ldg(reinterpret_cast<const uint4*>(src) + v);
      gw[i] = __ldg(reinterpret_cast<const uint4*>(gamma) + v);
      sm[2 * i] = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v);
      sm[2 * i + 1] = __ldg(reinterpret_cast<const float4*>(smooth) + 2 * v + 1);
    }
  }
  float x[VPT][8];
  double ss = 0.0;
  bool wide = false;   // a value outside [2^-60, 2^60] (not zero): square this thread's values in fp64
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v >= nvec) continue;
    bf16x8_to_f32(raw[i], x[i]);
    float sg = 0.f, cg = 0.f;   // the group's running sum and the exact sum of its rounding errors
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t ex = (__float_as_uint(x[i][e]) >> 23) & 0xFFu;
      wide |= x[i][e] != 0.f && (ex < 127u - 60u || ex > 127u + 60u);
      const float y = __fmul_rn(x[i][e], x[i][e]);
      const float t = __fadd_rn(sg, y);
      cg = __fadd_rn(cg, __fadd_rn(__fsub_rn(fmaxf(sg, y), t), fminf(sg, y)));
      sg = t;
    }
    ss = __dadd_rn(ss, __dadd_rn((double)sg, (double)cg));
  }
  if (wide) {
    ss = 0.0;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = threadIdx.x + i * THREADS;
      if (v >= nvec) continue;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const double d = (double)x[i][e];
        ss = __dadd_rn(ss, __dmul_rn(d, d));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  __shared__ double red64[THREADS / 32];
  __shared__ float r_s;
  if ((threadIdx.x & 31) == 0) red64[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = red64[0];
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) t = __dadd_rn(t, red64[w]);
    const double ms = __ddiv_rn(t, (double)K);
    r_s = __double2float_rn(__ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(ms, (double)eps))));
  }
  __syncthreads();
  const float r = r_s;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v >= nvec) continue;
    float g[8];
    bf16x8_to_f32(gw[i], g);
    const float s[8] = {sm[2 * i].x, sm[2 * i].y, sm[2 * i].z, sm[2 * i].w,
                        sm[2 * i + 1].x, sm[2 * i + 1].y, sm[2 * i + 1].z, sm[2 * i + 1].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float h = bf16_round(__fmul_rn(bf16_round(__fmul_rn(x[i][e], r)), g[e]));
      x[i][e] = __fmul_rn(h, s[e]);
      amax = fmaxf(amax, fabsf(x[i][e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[THREADS / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
  int8_t* dst = q + (size_t)row * K;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v >= nvec) continue;
    uint32_t packed[2] = {0u, 0u};
    if (amax > 0.f) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int c = __float2int_rn(__fmul_rn(x[i][e], inv));
        c = max(-127, min(127, c));
        packed[e >> 2] |= (uint32_t)(c & 0xFF) << (8 * (e & 3));
      }
    }
    reinterpret_cast<uint2*>(dst)[v] = make_uint2(packed[0], packed[1]);
  }
}

// The GLU glue of long rows, one row per thread-block cluster of C CTAs: CTA
// r of the cluster takes values [r K/C, (r+1) K/C) of the row (at most
// 2048 VPT of them, VPT 8-value vectors per thread), so a few rows still fill
// the GPU.  The row's absmax is the largest of the C CTAs' partial maxima,
// read from each CTA's shared memory across the cluster; a max is exact in
// any order, so codes and scale are those of quant_act_kernel<*, true>.
QUASAR_DEVICE_INLINE float ld_cluster_f32(const float* local, uint32_t rank) {
  const uint32_t remote = map_to_rank(local, rank);
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

template <int VPT>
__global__ void __launch_bounds__(THREADS) glu_quant_cluster_kernel(const uint16_t* __restrict__ in, int ld,
                                                                    const float* __restrict__ smooth, int K, int C,
                                                                    int8_t* __restrict__ q,
                                                                    float* __restrict__ scale) {
  pdl_launch_dependents();
  pdl_wait();
  const int rank = (int)cluster_ctarank();
  const int row = (int)cluster_id_x();
  const int slice = K / C;                                   // a multiple of 8
  const int nvec = slice / 8;
  const uint16_t* src = in + (size_t)row * ld + (size_t)rank * slice;
  const float* sms = smooth + (size_t)rank * slice;
  uint4 raw[VPT], rawu[VPT];
  float4 sm[2 * VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v < nvec) {
      raw[i] = __ldg(reinterpret_cast<const uint4*>(src) + v);
      rawu[i] = __ldg(reinterpret_cast<const uint4*>(src + K) + v);
      sm[2 * i] = __ldg(reinterpret_cast<const float4*>(sms) + 2 * v);
      sm[2 * i + 1] = __ldg(reinterpret_cast<const float4*>(sms) + 2 * v + 1);
    }
  }
  float x[VPT][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v >= nvec) continue;
    bf16x8_to_f32(raw[i], x[i]);
    glu8(x[i], rawu[i]);
    const float s[8] = {sm[2 * i].x, sm[2 * i].y, sm[2 * i].z, sm[2 * i].w,
                        sm[2 * i + 1].x, sm[2 * i + 1].y, sm[2 * i + 1].z, sm[2 * i + 1].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[i][e] = __fmul_rn(x[i][e], s[e]);
      amax = fmaxf(amax, fabsf(x[i][e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[THREADS / 32];
  __shared__ float cta_amax;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = red[0];
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) a = fmaxf(a, red[w]);
    cta_amax = a;
  }
  // Every CTA's partial maximum is in its shared memory before any is read.
  cluster_sync_full();
  amax = 0.f;
  for (int r = 0; r < C; ++r) amax = fmaxf(amax, ld_cluster_f32(&cta_amax, (uint32_t)r));
  // Reads done: arrive now, wait before exiting so that no CTA's shared
  // memory goes away while another CTA of the cluster may still read it.
  cluster_arrive_relaxed();
  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  if (rank == 0 && threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
  int8_t* dst = q + (size_t)row * K + (size_t)rank * slice;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * THREADS;
    if (v >= nvec) continue;
    uint32_t packed[2] = {0u, 0u};
    if (amax > 0.f) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int c = __float2int_rn(__fmul_rn(x[i][e], inv));
        c = max(-127, min(127, c));
        packed[e >> 2] |= (uint32_t)(c & 0xFF) << (8 * (e & 3));
      }
    }
    reinterpret_cast<uint2*>(dst)[v] = make_uint2(packed[0], packed[1]);
  }
  cluster_wait();
}

// Cluster shape for a GLU row of K values: the smallest C in {2, 4, 8} that
// divides the row into 8-value vectors with at most 2048 * vpt values per
// CTA, trying vpt = 1 first; {0, 0} when rows of K <= 2048 fit one CTA's
// single vector per thread, or no shape fits.
struct GluCluster {
  int C, vpt;
};
static GluCluster glu_cluster(int K) {
  if (K <= 2048) return {0, 0};
  for (int vpt = 1; vpt <= 2; ++vpt)
    for (int C = 2; C <= 8; C *= 2)
      if (K % (8 * C) == 0 && K / C <= 2048 * vpt) return {C, vpt};
  return {0, 0};
}

// Row-major INT8 codes [N][K] -> packed layout, 16 bytes per thread.
__global__ void tile_weights_kernel(const int8_t* __restrict__ src, int N, int K, int8_t* __restrict__ dst) {
  const int chunks = K / 16;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)N * chunks) return;
  const int n = (int)(i / chunks), k = (int)(i % chunks) * 16;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + (size_t)n * K + k));
  const uint32_t b = 0x80808080u;  // packed bytes hold code + 128
  *reinterpret_cast<uint4*>(dst + packed_offset(n, k, (K + 127) >> 7)) = make_uint4(v.x ^ b, v.y ^ b, v.z ^ b, v.w ^ b);
}

// ---- 4-bit weights.  Byte offset of 16-byte chunk c (K values 32c .. 32c+31
// of a block) of packed row n: blocks of 128 rows x 128 K are 8 KB, row r
// at 64 r, chunk c at (c ^ ((r >> 1) & 3)) * 16.  Byte j = 4 w + b of a
// chunk holds code(32c + 4w + b) + 8 in its low nibble and
// code(32c + 16 + 4w + b) + 8 in its high nibble.
QUASAR_DEVICE_INLINE size_t packed4_offset(int n, int k32, int KB) {
  const int r = n & 127, c = (k32 & 127) >> 5;
  return (((size_t)(n >> 7) * KB + (k32 >> 7)) * 128 + r) * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

// Sixteen packed bytes from the 32 codes of one chunk (missing K: code 0).
QUASAR_DEVICE_INLINE uint4 pack4_chunk(const int (&code)[32]) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t v = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t lo = (uint32_t)(code[4 * q + b] + 8) & 0xF, hi = (uint32_t)(code[16 + 4 * q + b] + 8) & 0xF;
      v |= (lo | (hi << 4)) << (8 * b);
    }
    w[q] = v;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One CTA per weight row: w' = W / smooth, a = max |w'|, sw = a / 7,
// code = clamp(rne(w' * (7 / a)), -7, 7); the second pass packs 32 codes
// per thread step.
__global__ void __launch_bounds__(THREADS) quant_rows_w4_kernel(const uint16_t* __restrict__ in, int ld,
                                                                const float* __restrict__ smooth, int K,
                                                                int8_t* __restrict__ q, float* __restrict__ scale) {
  const int row = blockIdx.x;
  const uint16_t* src = in + (size_t)row * ld;
  float amax = 0.f;
  for (int k = threadIdx.x; k < K; k += THREADS)
    amax = fmaxf(amax, fabsf(__fdiv_rn(__uint_as_float((uint32_t)src[k] << 16), smooth[k])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[THREADS / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? __fdiv_rn(7.f, amax) : 0.f;
  if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 7.f) : 0.f;
  const int KB = (K + 127) >> 7;
  for (int k32 = 32 * threadIdx.x; k32 < K; k32 += 32 * THREADS) {
    int code[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int k = k32 + i;
      int c = 0;
      if (k < K && amax > 0.f) {
        c = __float2int_rn(__fmul_rn(__fdiv_rn(__uint_as_float((uint32_t)src[k] << 16), smooth[k]), inv));
        c = max(-7, min(7, c));
      }
      code[i] = c;
    }
    *reinterpret_cast<uint4*>(q + packed4_offset(row, k32, KB)) = pack4_chunk(code);
  }
}

// Row-major codes [N][K] in [-8, 7] -> 4-bit packed layout, one chunk per thread.
__global__ void tile_weights_w4_kernel(const int8_t* __restrict__ src, int N, int K, int8_t* __restrict__ dst) {
  const int chunks = (K + 31) / 32;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)N * chunks) return;
  const int n = (int)(i / chunks), k32 = (int)(i % chunks) * 32;
  int code[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) code[j] = k32 + j < K ? (int)src[(size_t)n * K + k32 + j] : 0;
  *reinterpret_cast<uint4*>(dst + packed4_offset(n, k32, (K + 127) >> 7)) = pack4_chunk(code);
}

size_t packed_bytes(int N, int K) {
  if (N <= 0 || K <= 0) return 0;
  return (size_t)((N + 127) / 128) * ((K + 127) / 128) * 128 * 128;
}

// GLU: rows of [gate (K values) | up (K values)], quantizing silu(gate) * up
// (activations only: not with DIVIDE or PACKED).
template <bool DIVIDE, bool PACKED, bool GLU = false>
static quasar_status_t run(const void* in, int ld, const float* smooth, int rows, int K, int8_t* q, float* scale,
                           cudaStream_t stream, void* xh = nullptr) {
  static_assert(!(GLU && (DIVIDE || PACKED)), "the GLU glue is an activation step");
  if (rows < 0 || K <= 0 || (GLU && K > (1 << 29))) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || ld < (GLU ? 2 * K : K) || ld % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (rows == 0) return QUASAR_OK;  // empty batch: nothing is read or written
  if (!in || !smooth || !q || !scale) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(in, 16) || !aligned(smooth, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return QUASAR_ERR_UNSUPPORTED;
  if (PACKED) {
    // The padding of the last row tile and K block must read as zero codes
    // (byte 0x80 in the biased packed format).
    cudaError_t e = cudaMemsetAsync(q, 0x80, packed_bytes(rows, K), stream);
    if (e != cudaSuccess) return cuda_status(e);
    quant_rows_kernel<DIVIDE, PACKED><<<rows, THREADS, 0, stream>>>(reinterpret_cast<const uint16_t*>(in), ld,
                                                                    smooth, K, q, scale);
    return cuda_status(cudaGetLastError());
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(THREADS);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint16_t* x = reinterpret_cast<const uint16_t*>(in);
  if constexpr (GLU) {
    const GluCluster gc = glu_cluster(K);
    if (gc.C > 1) {
      cudaLaunchAttribute cattr[2];
      cattr[0] = attr[0];
      cattr[1].id = cudaLaunchAttributeClusterDimension;
      cattr[1].val.clusterDim.x = (unsigned)gc.C;
      cattr[1].val.clusterDim.y = 1;
      cattr[1].val.clusterDim.z = 1;
      cudaLaunchConfig_t ccfg = cfg;
      ccfg.gridDim = dim3((unsigned)rows * (unsigned)gc.C);
      ccfg.attrs = cattr;
      ccfg.numAttrs = 2;
      if (gc.vpt == 1)
        return cuda_status(cudaLaunchKernelEx(&ccfg, glu_quant_cluster_kernel<1>, x, ld, smooth, K, gc.C, q, scale));
      return cuda_status(cudaLaunchKernelEx(&ccfg, glu_quant_cluster_kernel<2>, x, ld, smooth, K, gc.C, q, scale));
    }
  }
  const int vpt = (K / 8 + THREADS - 1) / THREADS;   // 8-value vectors per thread
  uint4* xh4 = reinterpret_cast<uint4*>(xh);
  if (!DIVIDE && vpt <= 2)
    return cuda_status(cudaLaunchKernelEx(&cfg, quant_act_kernel<2, GLU>, x, ld, smooth, K, q, scale, xh4));
  if (!DIVIDE && vpt <= 6)
    return cuda_status(cudaLaunchKernelEx(&cfg, quant_act_kernel<6, GLU>, x, ld, smooth, K, q, scale, xh4));
  if (xh) return QUASAR_ERR_UNSUPPORTED;  // rows too long for the one-pass kernel: no fp16 copy
  return cuda_status(cudaLaunchKernelEx(&cfg, quant_rows_kernel<DIVIDE, PACKED, GLU>, x, ld, smooth, K, q, scale));
}

// Smooth + quantize (quasar_smooth_quant_act) and also write the codes as
// fp16 into `xh` [M][K]; QUASAR_ERR_UNSUPPORTED (nothing launched) when K is
// beyond the one-pass kernel's rows.
quasar_status_t smooth_quant_act_f16(const void* X_bf16, int ldx, const float* smooth, int M, int K, int8_t* Xq,
                                     float* sa, void* xh, cudaStream_t stream) {
  if (!xh || !aligned(xh, 16)) return QUASAR_ERR_INVALID_ARG;
  if ((K / 8 + THREADS - 1) / THREADS > 6) return QUASAR_ERR_UNSUPPORTED;
  return run<false, false>(X_bf16, ldx, smooth, M, K, Xq, sa, stream, xh);
}

}  // namespace quant
}  // namespace quasar

extern "C" {

size_t quasar_packed_weight_bytes(int N, int K) { return quasar::quant::packed_bytes(N, K); }

quasar_status_t quasar_pack_weights(const void* W_bf16, int ldw, const float* smooth, int N, int K, int8_t* Wp,
                                    float* sw, quasar_stream_t stream) {
  if (N <= 0) return QUASAR_ERR_INVALID_ARG;
  return quasar::quant::run<true, true>(W_bf16, ldw, smooth, N, K, Wp, sw, reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_tile_weights(const int8_t* Wq, int N, int K, int8_t* Wp, quasar_stream_t stream_) {
  using namespace quasar;
  if (N <= 0 || K <= 0 || !Wq || !Wp) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (!aligned(Wq, 16) || !aligned(Wp, 16)) return QUASAR_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaMemsetAsync(Wp, 0x80, quant::packed_bytes(N, K), stream);
  if (e != cudaSuccess) return cuda_status(e);
  const long long items = (long long)N * (K / 16);
  quant::tile_weights_kernel<<<(unsigned)((items + 255) / 256), 256, 0, stream>>>(Wq, N, K, Wp);
  return cuda_status(cudaGetLastError());
}

size_t quasar_packed_weight_bytes_w4(int N, int K) { return quasar::quant::packed_bytes(N, K) / 2; }

quasar_status_t quasar_pack_weights_w4(const void* W_bf16, int ldw, const float* smooth, int N, int K, int8_t* Wp4,
                                       float* sw, quasar_stream_t stream_) {
  using namespace quasar;
  if (N < 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || ldw < K || ldw % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (N == 0) return QUASAR_OK;
  if (!W_bf16 || !smooth || !Wp4 || !sw) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(W_bf16, 16) || !aligned(smooth, 4) || !aligned(Wp4, 16) || !aligned(sw, 4)) return QUASAR_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaMemsetAsync(Wp4, 0x88, quant::packed_bytes(N, K) / 2, stream);   // padding: code 0
  if (e != cudaSuccess) return cuda_status(e);
  quant::quant_rows_w4_kernel<<<N, quant::THREADS, 0, stream>>>(reinterpret_cast<const uint16_t*>(W_bf16), ldw, smooth,
                                                                 K, Wp4, sw);
  return cuda_status(cudaGetLastError());
}

quasar_status_t quasar_tile_weights_w4(const int8_t* Wq4, int N, int K, int8_t* Wp4, quasar_stream_t stream_) {
  using namespace quasar;
  if (N <= 0 || K <= 0 || !Wq4 || !Wp4) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (!aligned(Wp4, 16)) return QUASAR_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaMemsetAsync(Wp4, 0x88, quant::packed_bytes(N, K) / 2, stream);
  if (e != cudaSuccess) return cuda_status(e);
  const long long items = (long long)N * ((K + 31) / 32);
  quant::tile_weights_w4_kernel<<<(unsigned)((items + 255) / 256), 256, 0, stream>>>(Wq4, N, K, Wp4);
  return cuda_status(cudaGetLastError());
}

quasar_status_t quasar_smooth_quant_act(const void* X_bf16, int ldx, const float* smooth, int M, int K,
                                        int8_t* Xq, float* sa, quasar_stream_t stream) {
  return quasar::quant::run<false, false>(X_bf16, ldx, smooth, M, K, Xq, sa,
                                          reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_rmsnorm_smooth_quant(const void* X_bf16, int ldx, const void* gamma_bf16, float eps,
                                            const float* smooth, int M, int K, int8_t* Xq, float* sa,
                                            quasar_stream_t stream_) {
  using namespace quasar;
  if (M < 0 || K <= 0 || !(eps > 0.f) || !(eps < 3.0e38f)) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || ldx < K || ldx % 8 != 0 || K > 2048 * 6) return QUASAR_ERR_UNSUPPORTED;
  if (M == 0) return QUASAR_OK;
  if (!X_bf16 || !gamma_bf16 || !smooth || !Xq || !sa) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(X_bf16, 16) || !aligned(gamma_bf16, 16) || !aligned(smooth, 16) || !aligned(Xq, 16) ||
      !aligned(sa, 4))
    return QUASAR_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(quant::THREADS);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint16_t* x = reinterpret_cast<const uint16_t*>(X_bf16);
  const uint16_t* g = reinterpret_cast<const uint16_t*>(gamma_bf16);
  if (K / 8 <= 2 * quant::THREADS)
    return cuda_status(cudaLaunchKernelEx(&cfg, quant::rms_quant_kernel<2>, x, ldx, g, eps, smooth, K, Xq, sa));
  return cuda_status(cudaLaunchKernelEx(&cfg, quant::rms_quant_kernel<6>, x, ldx, g, eps, smooth, K, Xq, sa));
}

quasar_status_t quasar_silu_mul_smooth_quant(const void* GU_bf16, int ldgu, const float* smooth, int M, int I,
                                             int8_t* Xq, float* sa, quasar_stream_t stream) {
  return quasar::quant::run<false, false, true>(GU_bf16, ldgu, smooth, M, I, Xq, sa,
                                                reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
