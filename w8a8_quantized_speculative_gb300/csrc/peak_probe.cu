// Tensor-pipe rate probe: how fast the MMA forms that the W8A8 kernels use
// run on this device, so that tensor-pipe fractions are quoted against a
// measured rate of the same instruction rather than a datasheet figure.
//
// sm_103a has no integer tcgen05 MMA (kind::i8 is rejected for this target),
// so the INT8 codes run on the fp16 path: tcgen05.mma kind::f16 with fp32
// accumulators in TMEM (the tcgen05 kernel, weights as the A operand in
// TMEM), and the warp-level mma.sync m16n8k16 (the register-path kernel).
//
// Forms (one CTA per SM, every SM measured):
//   0  tcgen05.mma kind::f16, M = 128, N = n, K = 16, A in TMEM, B in shared
//      memory, back-to-back into one accumulator
//   1  the same with A in shared memory (128B-swizzled, K-major)
//   2  form 0 while 16 other warps store into another TMEM region with
//      tcgen05.st (the converters' traffic in the W8A8 kernel)
//   3  mma.sync.m16n8k16 f16 x f16 -> f32 from registers, 16 warps, four
//      independent accumulator chains per warp
//   4, 5  form 0 with the four K steps of each group spread over two / four
//      independent accumulators (N <= 128): whether separate accumulation
//      chains overlap in the tensor pipe
//   6  form 1 with M = 64 (64 A rows in shared memory)
//   7  tcgen05.mma.cta_group::2 kind::f16, M = 256 over a cluster of two
//      CTAs on two SMs (128 A rows in each CTA's TMEM), N = n (n / 2 B rows
//      in each CTA's shared memory), K = 16, issued by the even CTA
//   8  form 7 with A in shared memory
// Each CTA records its cycle count (clock64) and the work it issued (in the
// pair forms the issuing CTA records for both SMs: each does 128 x n x 16
// MACs per instruction).
#include "quasar_common.cuh"

namespace quasar {
namespace probe {

constexpr int WARPS = 18;           // warp 0: TMEM + MMA issue; 1-16: tcgen05.st traffic; 17: idle
constexpr int D_COL = 0;            // accumulator columns [0, n)
constexpr int A_COL = 256;          // A operand (form 0 / 2): 64 K as 32 columns of fp16 pairs
constexpr int NOISE_COL = 384;      // tcgen05.st traffic region: 4 x 16 columns
constexpr int SMEM_A = 16384;       // 128 rows x 64 K fp16, 128B-swizzled
constexpr int SMEM_B = 32768;       // up to 256 rows x 64 K fp16
constexpr int SMEM_USED = 1024 + SMEM_A + SMEM_B + 64;
// Requested per CTA so that no two probe CTAs share an SM (each allocates all
// 512 TMEM columns and each SM's rate is measured alone).
constexpr int SMEM_BYTES = 120 * 1024;
static_assert(SMEM_USED <= SMEM_BYTES, "probe shared memory");

QUASAR_DEVICE_INLINE uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// out[blockIdx.x * 4 + {0,1,2,3}] = cycles of the MMA loop, MMAs issued,
// tcgen05.st instructions completed by the traffic warps, cycles they ran.
__global__ void __launch_bounds__(32 * WARPS, 1)
tc_probe_kernel(int form, int n, int iters, unsigned long long* out, unsigned int* err,
                unsigned long long limit_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + SMEM_A;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sb + SMEM_B);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* done = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* abort_flag = done + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // operands: zeros (the rate does not depend on the values)
  for (int i = threadIdx.x; i < (SMEM_A + SMEM_B) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *done = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 1 && warp <= 4) {   // zero the A region; a warp reaches TMEM lanes 32 (warp % 4) .. +31 only
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0;
    tmem_st32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + A_COL, z);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t mrows = form == 6 ? 64u : 128u;
      const uint32_t idesc = (1u << 4) | (uint32_t(n >> 3) << 17) | ((mrows >> 4) << 24);
      const uint64_t bdesc = desc_sw128(smem_u32(sb));
      const uint64_t adesc = desc_sw128(smem_u32(sa));
      const unsigned long long t0 = clock64();
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chains = form == 4 ? 2 : form == 5 ? 4 : 1;
          const uint32_t dcol = D_COL + (uint32_t)((k % chains) * n);
          const uint32_t acc = (it | (k / chains)) ? 1u : 0u;
          if (form == 1 || form == 6) {
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem + D_COL),
                "l"(adesc + (uint64_t)(2 * k)), "l"(bdesc + (uint64_t)(2 * k)), "r"(idesc), "r"(acc)
                : "memory");
          } else {
            tc_mma_f16_ts(tmem + dcol, tmem + A_COL + 8 * k, bdesc + (uint64_t)(2 * k), idesc, acc);
          }
        }
      }
      tc_commit(bar);
      const bool ok = mbar_wait(bar, 0, abort_flag, err, SITE_SELFTEST, limit_ns);
      const unsigned long long t1 = clock64();
      out[blockIdx.x * 4 + 0] = ok ? t1 - t0 : 0ull;
      out[blockIdx.x * 4 + 1] = (unsigned long long)iters * 4;
      *done = 1;
    }
    __syncwarp();
  } else if (warp <= 16 && form == 2) {
    // tcgen05.st traffic until the MMA loop is done (bounded)
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = (uint32_t)i;
    // warps 1-16: lane quadrant warp % 4, column group (warp - 1) / 4
    const uint32_t addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + NOISE_COL + 16 * ((warp - 1) >> 2);
    unsigned long long cnt = 0;
    const unsigned long long t0 = clock64();
    for (int i = 0; i < (1 << 22); ++i) {
      tmem_st16(addr, z);
      tc_wait_st();
      ++cnt;
      if (__shfl_sync(0xffffffffu, *done, 0)) break;
    }
    const unsigned long long t1 = clock64();
    if (lane == 0) {
      atomicAdd(&out[blockIdx.x * 4 + 2], cnt);
      atomicMax(&out[blockIdx.x * 4 + 3], t1 - t0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---- two-CTA (cta_group::2) forms
// TMEM allocation and release are collective over the pair (one warp of
// each CTA; both get the same address).
QUASAR_DEVICE_INLINE void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
QUASAR_DEVICE_INLINE void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
QUASAR_DEVICE_INLINE void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Completion of the pair MMAs this thread issued arrives on the barrier at
// the same offset in each CTA of `mask` (bit r: cluster rank r).
QUASAR_DEVICE_INLINE void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// The pair kernel takes 256 TMEM columns per CTA: accumulators [0, n), the
// TMEM A operand (form 7) at PAIR_A_COL; two allocations of that size fit in
// an SM's 512 columns whichever CTA's request covers which SM.
constexpr int PAIR_COLS = 256;
constexpr int PAIR_A_COL = 224;

__global__ void __launch_bounds__(32 * WARPS, 1)
tc_pair_probe_kernel(int form, int n, int iters, unsigned long long* out, unsigned int* err,
                     unsigned long long limit_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + SMEM_A;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sb + SMEM_B);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  for (int i = threadIdx.x; i < (SMEM_A + SMEM_B) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc_pair(tmem_slot, PAIR_COLS);
  tc_fence_before();
  cluster_sync_full();   // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  if (warp == 0) tmem_relinquish_pair();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) out[blockIdx.x * 4 + 2] = tmem;   // the TMEM address this CTA's request returned
  if (form == 7 && warp >= 1 && warp <= 4) {
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0;
    tmem_st32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + PAIR_A_COL, z);
    tc_wait_st();
  }
  tc_fence_before();
  cluster_sync_full();   // both CTAs' operands in place
  tc_fence_after();

  if (warp == 0) {
    if (lane == 0) {
      if (rank == 0) {
        const uint32_t idesc = (1u << 4) | (uint32_t(n >> 3) << 17) | ((256u >> 4) << 24);
        const uint64_t bdesc = desc_sw128(smem_u32(sb));
        const uint64_t adesc = desc_sw128(smem_u32(sa));
        const unsigned long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (it | k) ? 1u : 0u;
            if (form == 8)
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem + D_COL),
                  "l"(adesc + (uint64_t)(2 * k)), "l"(bdesc + (uint64_t)(2 * k)), "r"(idesc), "r"(acc)
                  : "memory");
            else
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + D_COL),
                  "r"(tmem + PAIR_A_COL + 8 * k), "l"(bdesc + (uint64_t)(2 * k)), "r"(idesc), "r"(acc)
                  : "memory");
          }
        }
        tc_commit_pair(bar, 3);
        const bool ok = mbar_wait(bar, 0, abort_flag, err, SITE_SELFTEST, limit_ns);
        const unsigned long long t1 = clock64();
        out[blockIdx.x * 4 + 0] = ok ? t1 - t0 : 0ull;
        out[blockIdx.x * 4 + 1] = (unsigned long long)iters * 4;
      } else {
        // the even CTA's commit arrives here as well; its MMAs write this
        // CTA's TMEM, so wait for them before releasing it
        mbar_wait(bar, 0, abort_flag, err, SITE_SELFTEST, limit_ns);
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  cluster_sync_full();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, PAIR_COLS);
  }
}

// D += A * B, m16n8k16 fp16 -> fp32 from registers.
QUASAR_DEVICE_INLINE void hmma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// out[blockIdx.x * 4 + 0] = cycles of the slowest warp, [1] = MMAs issued by the CTA.
__global__ void __launch_bounds__(512, 1) hmma_probe_kernel(int iters, unsigned long long* out, float* sink) {
  float d[4][4] = {};
  const uint32_t a = 0x3c003c00u, b = 0x3c003c00u;   // fp16 ones: finite sums
  const unsigned long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < 4; ++c) hmma(d[c], a, a, a, a, b, b);
  }
  const unsigned long long t1 = clock64();
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&out[blockIdx.x * 4 + 0], t1 - t0);
    atomicAdd(&out[blockIdx.x * 4 + 1], (unsigned long long)iters * 4);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
  if (s == 1234.5f) sink[threadIdx.x] = s;   // keeps the MMAs live; never true for these inputs
}

}  // namespace probe
}  // namespace quasar

extern "C" quasar_status_t quasar_probe_tensor_rate(int form, int n, int iters, unsigned long long* out,
                                                    int out_slots, quasar_stream_t stream_) {
  using namespace quasar;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!out || iters <= 0 || iters > (1 << 20)) return QUASAR_ERR_INVALID_ARG;
  if (form < 0 || form > 8) return QUASAR_ERR_INVALID_ARG;
  if (form != 3 && (n < 16 || n > 256 || n % 16 != 0)) return QUASAR_ERR_UNSUPPORTED;
  if ((form == 4 && n > 128) || (form == 5 && n > 64)) return QUASAR_ERR_UNSUPPORTED;   // accumulators below A_COL
  if (form == 7 && n > probe::PAIR_A_COL) return QUASAR_ERR_UNSUPPORTED;                // accumulator below the A operand
  const int sms = sm_count();
  if (sms <= 0) return QUASAR_ERR_CUDA;
  if (out_slots < 4 * sms) return QUASAR_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(out, 0, (size_t)4 * sms * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return cuda_status(e);
  if (form == 3) {
    static int hconf[64] = {0};
    int hdev = 0;
    cudaGetDevice(&hdev);
    if (hdev >= 0 && hdev < 64 && !hconf[hdev]) {
      e = cudaFuncSetAttribute(probe::hmma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               probe::SMEM_BYTES);
      if (e != cudaSuccess) return cuda_status(e);
      hconf[hdev] = 1;
    }
    probe::hmma_probe_kernel<<<sms, 512, probe::SMEM_BYTES, stream>>>(iters, out, reinterpret_cast<float*>(out));
    return cuda_status(cudaGetLastError());
  }
  unsigned int* err = device_error_word();
  if (!err) return QUASAR_ERR_CUDA;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(probe::tc_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, probe::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    configured[dev] = 1;
  }
  if (form == 7 || form == 8) {
    static int pconf[64] = {0};
    if (dev >= 0 && dev < 64 && !pconf[dev]) {
      e = cudaFuncSetAttribute(probe::tc_pair_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               probe::SMEM_BYTES);
      if (e != cudaSuccess) return cuda_status(e);
      pconf[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms / 2 * 2));
    cfg.blockDim = dim3(32 * probe::WARPS);
    cfg.dynamicSmemBytes = probe::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, probe::tc_pair_probe_kernel, form, n, iters, out, err,
                                          wait_limit_ns()));
  }
  probe::tc_probe_kernel<<<sms, 32 * probe::WARPS, probe::SMEM_BYTES, stream>>>(form, n, iters, out, err,
                                                                                 wait_limit_ns());
  return cuda_status(cudaGetLastError());
}
