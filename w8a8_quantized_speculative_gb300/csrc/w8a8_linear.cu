// A3 + A4: W8A8 verify linear on sm_103a.
//
//   acc[m][n] = sum_k Xq[m][k] * Wq[n][k]        exact integer
//   Y[m][n]   = bf16_rne((float(acc) * sa[m]) * sw[n])
//
// Quasar summary pt §2 "Metodologia" steps 3-4: the matmul runs on INT8
// operands and the result is dequantized to BF16 before the nonlinear
// layers.  In a verification pass M = batch x (drafts + 1) is small and the
// INT8 weight stream from HBM sets the time (pt §1, zh §1: verification is
// memory-bandwidth bound).
//
// Design (GB300-native):
//  * sm_103a has no tcgen05 integer MMA, so INT8 codes are widened to fp16
//    (exact for |v| <= 2048) and multiplied with tcgen05.mma kind::f16 into
//    fp32 accumulators in TMEM.  Products are <= 127^2 = 16129 < 2^14 and an
//    accumulation run is capped at K = 1024, so every partial sum is an
//    integer below 16129*1024 < 2^24 and fp32 holds it exactly.  Each run is
//    drained to int32 registers (cvt.rni), so the result is the exact
//    integer sum for any K.
//  * Swap-AB: weight rows fill the MMA's M = 128 side, tokens the N side
//    (NT = 16..128).  The weight tile is the A operand and lives in TMEM:
//    converter warps read the TMA-staged INT8 tile from shared memory, widen
//    it in registers and tcgen05.st it into TMEM.  Shared memory then carries
//    ~2 bytes per weight (TMA write + one read) instead of the ~6 a widened
//    shared-memory A operand would cost.  The small token tile is widened
//    into a 128B-swizzled K-major shared-memory B operand.
//  * Persistent grid of one CTA per SM.  The (weight tile, 128-wide K block)
//    work list is split into equal contiguous ranges, one per CTA (stream-K
//    style), so every SM streams the same number of weight bytes.  A CTA whose
//    range covers a whole tile writes Y directly; partial tiles are summed
//    with integer atomics (order-independent, so still exact and
//    deterministic) into a zero-filled workspace.  Each converter warp owns
//    the same 32-row x NT/2-token sub-tile in every CTA, so completion is
//    counted per (tile, warp): the warp whose K-block count completes the
//    sub-tile (no warp ever waits on another CTA) applies the epilogue and
//    re-zeroes the workspace slice and counter it used.
//  * Warp roles: warps 0-7 convert (and drain / run the epilogue), warp 8
//    issues TMA, warp 9 allocates TMEM and issues MMAs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "quasar_common.cuh"

namespace quasar {
namespace gemm {

constexpr int BM = 128;        // weight rows per tile (MMA M)
constexpr int BK = 128;        // K per block (bytes of INT8 = one 128B swizzle row)
constexpr int RUN_MAX = 8;     // blocks per fp32 accumulation run: K <= 1024 stays exact
constexpr int CONV_WARPS = 8;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 512;

template <int NT>
struct Cfg {
  static constexpr int S2 = (NT == 128) ? 3 : 4;            // converted stages (TMEM A + smem B)
  static constexpr int W_BYTES = BM * BK;                    // 16 KB INT8 weight tile
  static constexpr int X_BYTES = NT * BK;                    // INT8 token tile
  static constexpr int STAGE1 = W_BYTES + X_BYTES;           // multiple of 1024
  static constexpr int B16_BYTES = NT * BK * 2;              // fp16 token tile, 2 swizzle atoms
  static constexpr int S1 = (NT == 16) ? 8 : (NT == 32) ? 8 : (NT == 64) ? 6 : 3;  // INT8 stages
  static constexpr int A_COLS = BK / 2;                      // TMEM columns per A stage (fp16 pairs)
  static constexpr int TMEM_A0 = 2 * NT;                     // A stages follow two accumulators
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + S1 * STAGE1 + S2 * B16_BYTES + BAR_BYTES;
  static_assert(TMEM_A0 + S2 * A_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(STAGE1 % 1024 == 0 && B16_BYTES % 1024 == 0, "1024B alignment of swizzled tiles");
  static_assert(SMEM <= 232448, "shared memory budget");
  // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A/B fp16
  // (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
  static constexpr uint32_t IDESC = (1u << 4) | (uint32_t(NT >> 3) << 17) | (uint32_t(BM >> 4) << 24);
};

struct Params {
  const float* sa;
  const float* sw;
  int M, N, K;
  int KB;          // K blocks per tile
  int m_tiles;     // token tiles of NT
  int tiles;       // n_tiles * m_tiles
  long long total; // tiles * KB
  __nv_bfloat16* Y;
  int ldy;
  int32_t* acc_out;   // int32 mode when non-null
  int32_t* ws_acc;    // [M][N] int32, zero between calls
  uint32_t* ws_cnt;   // [tiles][8] K-block counters per converter warp, zero between calls
  unsigned int* err;
  unsigned long long limit_ns;
};

// Shared-memory matrix descriptor for a 128B-swizzled K-major tile whose
// 8-row groups are 1024 bytes apart (tcgen05 descriptor format: start >> 4
// in bits 0-13, leading offset (unused for swizzled K-major) in 16-29,
// stride offset >> 4 in 32-45, version 1 in bits 46-47, swizzle mode 2 =
// 128B in bits 61-63).
QUASAR_DEVICE_INLINE uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

template <int NT>
QUASAR_DEVICE_INLINE void tmem_ld_acc(uint32_t taddr, int32_t (&acc)[NT / 2]) {
  // Drain NT/2 fp32 accumulator columns in groups of 8; each holds an exact
  // integer, converted with round-to-nearest (no rounding actually occurs).
#pragma unroll
  for (int g = 0; g < NT / 16; ++g) {
    uint32_t v[8];
    tmem_ld8(taddr + g * 8, v);
    tc_wait_ld();
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[g * 8 + j] += __float2int_rn(__uint_as_float(v[j]));
  }
}

template <int NT>
__global__ void __launch_bounds__(THREADS, 1)
w8a8_linear_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const Params p) {
  using C = Cfg<NT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage1 = smem;                                  // S1 x [W 16KB | X NT*128]
  uint8_t* b16 = smem + C::S1 * C::STAGE1;                 // S2 x [2 atoms][NT][128B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(b16 + C::S2 * C::B16_BYTES);
  uint64_t* full1 = bars;                     // [S1] TMA -> converters
  uint64_t* empty1 = full1 + C::S1;           // [S1] converters -> TMA
  uint64_t* full2 = empty1 + C::S1;           // [S2] converters -> MMA
  uint64_t* empty2 = full2 + C::S2;           // [S2] MMA -> converters
  uint64_t* accfull = empty2 + C::S2;         // [2]  MMA -> drain
  uint64_t* accempty = accfull + 2;           // [2]  drain -> MMA
  uint64_t* mma_done = accempty + 2;          // [1]  final MMA drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S1; ++s) { mbar_init(&full1[s], 1); mbar_init(&empty1[s], CONV_WARPS); }
    for (int s = 0; s < C::S2; ++s) { mbar_init(&full2[s], CONV_WARPS); mbar_init(&empty2[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&accfull[a], 1); mbar_init(&accempty[a], CONV_WARPS); }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This CTA's contiguous range of (tile, K block) work items.
  const long long b0 = (long long)blockIdx.x * p.total / gridDim.x;
  const long long b1 = (long long)(blockIdx.x + 1) * p.total / gridDim.x;
  const int KB = p.KB;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      long long li = 0;
      for (long long i = b0; i < b1; ++i, ++li) {
        const int s = (int)(li % C::S1);
        const uint32_t round = (uint32_t)(li / C::S1);
        if (round > 0 &&
            !mbar_wait(&empty1[s], (round - 1) & 1, abort_flag, p.err, SITE_GEMM_EMPTY1, p.limit_ns))
          break;
        const int t = (int)(i / KB), kb = (int)(i % KB);
        const int n_tile = t / p.m_tiles, m_tile = t % p.m_tiles;
        uint8_t* st = stage1 + s * C::STAGE1;
        mbar_arrive_expect_tx(&full1[s], C::STAGE1);
        tma_load_2d(st, &tmW, kb * BK, n_tile * BM, &full1[s], pol_w);
        tma_load_2d(st + C::W_BYTES, &tmX, kb * BK, m_tile * NT, &full1[s], pol_x);
      }
      // Never leave with copies in flight: wait for the last phase issued on
      // every stage (already complete in a normal run).
      const long long issued = li;
      for (int s = 0; s < C::S1 && s < issued; ++s) {
        const long long last_li = s + ((issued - 1 - s) / C::S1) * C::S1;
        const uint32_t round = (uint32_t)(last_li / C::S1);
        volatile int dummy = 0;
        mbar_wait(&full1[s], round & 1, &dummy, p.err, SITE_GEMM_DRAIN, p.limit_ns);
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      long long li = 0;
      int R = -1;
      bool ok = true;
      for (long long i = b0; i < b1 && ok; ++i, ++li) {
        const int t = (int)(i / KB), kb = (int)(i % KB);
        const long long seg_start = b0 > (long long)t * KB ? b0 : (long long)t * KB;
        const int pos = (int)(i - seg_start);
        const bool seg_last = (i == b1 - 1) || (kb == KB - 1);
        const bool run_first = (pos % RUN_MAX) == 0;
        const bool run_last = seg_last || (pos % RUN_MAX) == RUN_MAX - 1;
        if (run_first) {
          ++R;
          if (R >= 2 && !mbar_wait(&accempty[R & 1], ((R >> 1) - 1) & 1, abort_flag, p.err, SITE_GEMM_ACCEMPTY,
                                   p.limit_ns)) {
            ok = false;
            break;
          }
        }
        const int r = (int)(li % C::S2);
        if (!mbar_wait(&full2[r], (uint32_t)(li / C::S2) & 1, abort_flag, p.err, SITE_GEMM_FULL2, p.limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)((R & 1) * NT);
        const uint32_t a_tmem = tmem + (uint32_t)(C::TMEM_A0 + r * C::A_COLS);
        const uint32_t b_base = smem_u32(b16 + r * C::B16_BYTES);
#pragma unroll
        for (int k16 = 0; k16 < BK / 16; ++k16) {
          const uint64_t bdesc = sw128_kmajor_desc(b_base + (k16 >> 2) * (NT * 128) + (k16 & 3) * 32);
          tc_mma_f16_ts(d_tmem, a_tmem + k16 * 8, bdesc, C::IDESC, (run_first && k16 == 0) ? 0u : 1u);
        }
        tc_commit(&empty2[r]);
        if (run_last) tc_commit(&accfull[R & 1]);
      }
      // Wait until every MMA this thread issued has completed before the
      // CTA may release TMEM.
      tc_commit(mma_done);
      volatile int dummy = 0;
      mbar_wait(mma_done, 0, &dummy, p.err, SITE_GEMM_DRAIN, p.limit_ns);
    }
  } else {
    // ---------------------------------------------------------------- converters
    const int q = warp & 3;       // TMEM lane quadrant = weight rows 32q..32q+31
    const int h = warp >> 2;      // K half of the A tile; token half of the accumulator
    const int row = 32 * q + lane;
    const int ct = threadIdx.x;   // 0..255
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    int32_t acc[NT / 2];
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) acc[j] = 0;

    long long li = 0;
    int R = -1;
    for (long long i = b0; i < b1; ++i, ++li) {
      const int t = (int)(i / KB), kb = (int)(i % KB);
      const long long seg_start = b0 > (long long)t * KB ? b0 : (long long)t * KB;
      const int pos = (int)(i - seg_start);
      const bool seg_last = (i == b1 - 1) || (kb == KB - 1);
      const bool run_first = (pos % RUN_MAX) == 0;
      const bool run_last = seg_last || (pos % RUN_MAX) == RUN_MAX - 1;
      if (run_first) ++R;

      const int s = (int)(li % C::S1);
      const int r = (int)(li % C::S2);
      // Every lane waits; the warp then takes one decision, so the
      // .sync.aligned tcgen05 instructions below always see a full warp.
      bool ok = mbar_wait(&full1[s], (uint32_t)(li / C::S1) & 1, abort_flag, p.err, SITE_GEMM_FULL1, p.limit_ns);
      if (li >= C::S2)
        ok = ok && mbar_wait(&empty2[r], (uint32_t)((li / C::S2) - 1) & 1, abort_flag, p.err, SITE_GEMM_EMPTY2,
                             p.limit_ns);
      if (!__all_sync(0xffffffffu, ok)) break;

      const uint8_t* st = stage1 + s * C::STAGE1;
      // A: this thread's weight row, K half h (4 swizzled 16-byte chunks).
      {
        uint32_t a[32];
        const uint8_t* wrow = st + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * h + j;
          const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((c ^ (row & 7)) << 4));
          s8x4_to_f16x4(v.x, a[8 * j + 0], a[8 * j + 1]);
          s8x4_to_f16x4(v.y, a[8 * j + 2], a[8 * j + 3]);
          s8x4_to_f16x4(v.z, a[8 * j + 4], a[8 * j + 5]);
          s8x4_to_f16x4(v.w, a[8 * j + 6], a[8 * j + 7]);
        }
        tmem_st32(tmem + lane_off + (uint32_t)(C::TMEM_A0 + r * C::A_COLS + 32 * h), a);
      }
      // B: the token tile, NT rows x 8 chunks, widened into the swizzled fp16 tile.
      {
        const uint8_t* xs = st + C::W_BYTES;
        uint8_t* bd = b16 + r * C::B16_BYTES;
        for (int idx = ct; idx < NT * 8; idx += CONV_WARPS * 32) {
          const int xr = idx >> 3, c = idx & 7;
          const uint4 v = *reinterpret_cast<const uint4*>(xs + xr * 128 + ((c ^ (xr & 7)) << 4));
          uint4 o0, o1;
          s8x4_to_f16x4(v.x, o0.x, o0.y);
          s8x4_to_f16x4(v.y, o0.z, o0.w);
          s8x4_to_f16x4(v.z, o1.x, o1.y);
          s8x4_to_f16x4(v.w, o1.z, o1.w);
          uint8_t* dst = bd + (c >> 2) * (NT * 128) + xr * 128;
          const int cc = (c & 3) * 2;
          *reinterpret_cast<uint4*>(dst + ((cc ^ (xr & 7)) << 4)) = o0;
          *reinterpret_cast<uint4*>(dst + (((cc + 1) ^ (xr & 7)) << 4)) = o1;
        }
      }
      tc_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty1[s]);
        mbar_arrive(&full2[r]);
      }

      if (run_last) {
        const int a = R & 1;
        const bool okf = mbar_wait(&accfull[a], (uint32_t)(R >> 1) & 1, abort_flag, p.err, SITE_GEMM_ACCFULL,
                                   p.limit_ns);
        if (!__all_sync(0xffffffffu, okf)) break;
        tc_fence_after();
        tmem_ld_acc<NT>(tmem + lane_off + (uint32_t)(a * NT + h * (NT / 2)), acc);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[a]);
      }

      if (seg_last) {
        const int n_tile = t / p.m_tiles, m_tile = t % p.m_tiles;
        const int n = n_tile * BM + row;
        const int m0 = m_tile * NT + h * (NT / 2);
        const int kb0 = (int)(seg_start - (long long)t * KB);
        const bool whole = (kb0 == 0) && (kb == KB - 1);
        bool emit = whole;
        if (!whole) {
          // Split tile: publish this warp's 32 x NT/2 sub-tile with integer
          // atomics, then count the K blocks it covered.  The warp that
          // brings the (tile, warp) counter to KB owns the finished sums.
          if (n < p.N) {
#pragma unroll
            for (int j = 0; j < NT / 2; ++j)
              if (m0 + j < p.M) atomicAdd(&p.ws_acc[(size_t)(m0 + j) * p.N + n], acc[j]);
          }
          __threadfence();
          __syncwarp();
          uint32_t last = 0;
          if (lane == 0) {
            const uint32_t nb = (uint32_t)(kb - kb0 + 1);
            const uint32_t old = atomicAdd(&p.ws_cnt[(size_t)t * CONV_WARPS + warp], nb);
            last = (old + nb == (uint32_t)KB) ? 1u : 0u;
          }
          emit = __shfl_sync(0xffffffffu, last, 0) != 0;
          if (emit) {
            __threadfence();
            if (n < p.N) {
#pragma unroll
              for (int j = 0; j < NT / 2; ++j)
                if (m0 + j < p.M) acc[j] = atomicExch(&p.ws_acc[(size_t)(m0 + j) * p.N + n], 0);
            }
            if (lane == 0) atomicExch(&p.ws_cnt[(size_t)t * CONV_WARPS + warp], 0u);
          }
        }
        if (emit && n < p.N) {
          if (p.acc_out) {
#pragma unroll
            for (int j = 0; j < NT / 2; ++j)
              if (m0 + j < p.M) p.acc_out[(size_t)(m0 + j) * p.N + n] = acc[j];
          } else {
            const float swn = p.sw[n];
#pragma unroll
            for (int j = 0; j < NT / 2; ++j) {
              if (m0 + j < p.M) {
                const float y = __fmul_rn(__fmul_rn(__int2float_rn(acc[j]), p.sa[m0 + j]), swn);
                p.Y[(size_t)(m0 + j) * p.ldy + n] = __float2bfloat16_rn(y);
              }
            }
          }
        }
#pragma unroll
        for (int j = 0; j < NT / 2; ++j) acc[j] = 0;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

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

static bool encode_2d_u8(CUtensorMap* map, const void* base, int inner, int outer, int box_inner, int box_outer) {
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

static int pick_nt(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

struct Shape {
  int NT, m_tiles, n_tiles, tiles, KB;
};

static Shape shape_of(int M, int N, int K) {
  Shape s;
  s.NT = pick_nt(M);
  s.m_tiles = (M + s.NT - 1) / s.NT;
  s.n_tiles = (N + BM - 1) / BM;
  s.tiles = s.n_tiles * s.m_tiles;
  s.KB = (K + BK - 1) / BK;
  return s;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t workspace_size(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  Shape s = shape_of(M, N, K);
  return align256((size_t)s.tiles * CONV_WARPS * 4) + align256((size_t)M * N * 4);
}

template <int NT>
static cudaError_t launch_nt(const CUtensorMap& tw, const CUtensorMap& tx, const Params& p, int grid,
                             cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(w8a8_linear_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<NT>::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  w8a8_linear_kernel<NT><<<grid, THREADS, Cfg<NT>::SMEM, stream>>>(tw, tx, p);
  return cudaGetLastError();
}

quasar_status_t run(const int8_t* Xq, const float* sa, const int8_t* Wq, const float* sw, int M, int N, int K,
                    void* Y, int ldy, int32_t* acc_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 0 || N <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || N % 8 != 0 || K > 131072) return QUASAR_ERR_UNSUPPORTED;
  if (!acc_out && (ldy < N || ldy % 8 != 0)) return QUASAR_ERR_UNSUPPORTED;
  if (M == 0) return QUASAR_OK;  // empty batch: nothing is read or written
  if (!Xq || !Wq || (!acc_out && (!Y || !sa || !sw))) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(Xq, 16) || !aligned(Wq, 16) || (Y && !aligned(Y, 16)) || (acc_out && !aligned(acc_out, 16)) ||
      (sa && !aligned(sa, 4)) || (sw && !aligned(sw, 4)))
    return QUASAR_ERR_UNSUPPORTED;
  const size_t need = workspace_size(M, N, K);
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return QUASAR_ERR_WORKSPACE;

  Shape s = shape_of(M, N, K);
  CUtensorMap tw, tx;
  if (!encode_2d_u8(&tw, Wq, K, N, BK, BM)) return QUASAR_ERR_CUDA;
  if (!encode_2d_u8(&tx, Xq, K, M, BK, s.NT)) return QUASAR_ERR_CUDA;

  Params p;
  p.sa = sa;
  p.sw = sw;
  p.M = M;
  p.N = N;
  p.K = K;
  p.KB = s.KB;
  p.m_tiles = s.m_tiles;
  p.tiles = s.tiles;
  p.total = (long long)s.tiles * s.KB;
  p.Y = reinterpret_cast<__nv_bfloat16*>(Y);
  p.ldy = ldy;
  p.acc_out = acc_out;
  p.ws_cnt = reinterpret_cast<uint32_t*>(ws);
  p.ws_acc = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) + align256((size_t)s.tiles * CONV_WARPS * 4));
  p.err = device_error_word();
  p.limit_ns = wait_limit_ns();
  if (!p.err) return QUASAR_ERR_CUDA;

  const int sms = sm_count();
  if (sms <= 0) return QUASAR_ERR_CUDA;
  const int grid = (int)std::min<long long>(p.total, sms);
  cudaError_t e;
  switch (s.NT) {
    case 16: e = launch_nt<16>(tw, tx, p, grid, stream); break;
    case 32: e = launch_nt<32>(tw, tx, p, grid, stream); break;
    case 64: e = launch_nt<64>(tw, tx, p, grid, stream); break;
    default: e = launch_nt<128>(tw, tx, p, grid, stream); break;
  }
  return cuda_status(e);
}

}  // namespace gemm
}  // namespace quasar

extern "C" {

size_t quasar_w8a8_linear_workspace_size(int M, int N, int K) { return quasar::gemm::workspace_size(M, N, K); }

quasar_status_t quasar_w8a8_linear(const int8_t* Xq, const float* sa, const int8_t* Wq, const float* sw, int M,
                                   int N, int K, void* Y_bf16, int ldy, void* workspace, size_t ws_bytes,
                                   quasar_stream_t stream) {
  return quasar::gemm::run(Xq, sa, Wq, sw, M, N, K, Y_bf16, ldy, nullptr, workspace, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_int8_gemm_s32(const int8_t* Xq, const int8_t* Wq, int M, int N, int K, int32_t* acc,
                                     void* workspace, size_t ws_bytes, quasar_stream_t stream) {
  if (!acc && M > 0) return QUASAR_ERR_INVALID_ARG;
  return quasar::gemm::run(Xq, nullptr, Wq, nullptr, M, N, K, nullptr, 0, acc, workspace, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
