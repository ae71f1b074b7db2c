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
//    converter warps read the INT8 tile from shared memory, widen it in
//    registers and tcgen05.st it into TMEM.  Shared memory then carries ~2
//    bytes per weight (one bulk-copy write + one read) instead of the ~6 a
//    widened shared-memory A operand would cost.  The small token tile is
//    widened into a 128B-swizzled K-major shared-memory B operand.
//  * Weights arrive pre-packed (quasar_pack_weights) as contiguous 16 KB
//    blocks of 128 rows x 128 K, rows already in the 128B-swizzled order and
//    each code stored biased by +128, so one 1-D bulk copy per block streams
//    them from HBM and widening a byte takes no sign fix-up.  Tokens come
//    through a 2-D TMA tensor map.
//  * Persistent grid of one CTA per SM.  The (weight tile, K block) work list
//    is split into equal contiguous ranges, one per CTA (stream-K style), so
//    every SM streams the same number of weight bytes.  A CTA whose range
//    covers a whole tile writes Y directly; partial tiles are summed with
//    integer atomics (order-independent, so still exact and deterministic)
//    into a zero-filled workspace.  Each converter warp owns the same
//    32-row x NT/4-token sub-tile in every CTA, so completion is counted per
//    (tile, warp): the warp whose K-block count completes the sub-tile (no
//    warp ever waits on another CTA) applies the epilogue and re-zeroes the
//    workspace slice and counter it used.
//  * Programmatic dependent launch: the weight stream of the first stages
//    starts before the previous kernel in the stream has finished; token
//    loads and every global write wait for it (griddepcontrol.wait).
//  * Warp roles: warps 0-15 convert (and drain / run the epilogue), warp 16
//    issues the copies, warp 17 allocates TMEM and issues MMAs.
#include <algorithm>
#include <mutex>

#include "quasar_common.cuh"

namespace quasar {
namespace skinny {  // w8a8_skinny.cu: the register-path kernel, M <= 24 (skinny::handles)
bool handles(int M);
size_t slots_bytes(int M, int N, int K);
quasar_status_t run(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M, int N, int K,
                    void* Y, int ldy, int32_t* acc_out, uint32_t* ws_cnt, void* slots, cudaStream_t stream,
                    bool w4);
}  // namespace skinny

namespace quant {
quasar_status_t smooth_quant_act_f16(const void* X_bf16, int ldx, const float* smooth, int M, int K, int8_t* Xq,
                                     float* sa, void* xh, cudaStream_t stream);
}  // namespace quant

namespace gemm {

constexpr int BM = 128;        // weight rows per tile (MMA M)
constexpr int BK = 128;        // K per block (bytes of INT8 = one 128B swizzle row)
constexpr int RUN_MAX = 8;     // blocks per fp32 accumulation run: K <= 1024 stays exact
constexpr int CONV_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int WAITER_WARP = 18;
constexpr int THREADS = 32 * (CONV_WARPS + 3);
constexpr int MMA_BAR_ID = 1;   // named barrier pairing the MMA and waiter warps
constexpr int TMEM_COLS = 512;
constexpr int BLOCK_BYTES = BM * BK;   // one packed weight block

// XH: the token codes arrive already widened to fp16 (one copy per call in
// the workspace) and are copied by TMA straight into the MMA's B layout;
// the converters then widen only the weights, and the INT8 ring carries
// weight blocks alone.
template <int NT, bool XH = false>
struct Cfg {
  // Blocks per pipeline stage: two 128-K blocks per handshake halve the
  // per-byte cost of the barrier round trips; NT >= 96 keeps one (TMEM).
  static constexpr int G = (NT >= 96) ? 1 : 2;
  static constexpr int S2 = (NT >= 96) ? 3 : (NT == 64) ? 2 : 3;    // converted stages (TMEM A + smem B)
  static constexpr int W_BYTES = G * BLOCK_BYTES;            // INT8 weight blocks of a stage
  static constexpr int XB_BYTES = XH ? 0 : NT * BK;          // INT8 token tile of one block
  static constexpr int STAGE1 = W_BYTES + G * XB_BYTES;      // multiple of 1024
  static constexpr int B16_BLOCK = NT * BK * 2;              // fp16 token tile of one block (2 atoms)
  static constexpr int B16_BYTES = G * B16_BLOCK;
  // INT8 stages: as many as the shared memory holds next to the converted
  // stages (the pipeline is bound by copies in flight), at most 5.
  static constexpr int S1_FIT = (232448 - 1024 - 256 - S2 * G * NT * BK * 2) / (G * (BM * BK + XB_BYTES));
  static constexpr int S1 = XH ? (S1_FIT < 8 ? S1_FIT : 8)
                               : (NT == 16) ? 5 : (NT == 32) ? 4 : (NT == 64) ? 3 : (S1_FIT < 5 ? S1_FIT : 5);
  static constexpr int A_COLS = G * BK / 2;                  // TMEM columns per A stage (fp16 pairs)
  static constexpr int TMEM_A0 = 2 * NT;                     // A stages follow two accumulators
  static constexpr int TOK = NT / 4;                         // accumulator columns per converter thread
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + S1 * STAGE1 + S2 * B16_BYTES + BAR_BYTES;
  static_assert(RUN_MAX % G == 0, "stages never straddle an accumulation run");
  static_assert(TMEM_A0 + S2 * A_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(STAGE1 % 1024 == 0 && B16_BLOCK % 1024 == 0, "1024B alignment of swizzled tiles");
  static_assert(SMEM <= 232448, "shared memory budget");
  // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A/B fp16
  // (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
  static constexpr uint32_t IDESC = (1u << 4) | (uint32_t(NT >> 3) << 17) | (uint32_t(BM >> 4) << 24);
};

struct Params {
  const uint8_t* wp;  // packed weights, [n_tiles][KB][128 rows][128 B]
  const float* sa;
  const float* sw;
  int M, N, K;
  int KB;          // K blocks per tile
  int m_tiles;     // token tiles of NT
  int tiles;       // n_tiles * m_tiles
  int total;       // tiles * KB
  __nv_bfloat16* Y;
  int ldy;
  int32_t* acc_out;   // int32 mode when non-null
  int32_t* ws_acc;    // [M][N] int32, zero between calls
  uint32_t* ws_cnt;   // [tiles][16] K-block counters per converter warp, zero between calls
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

// Walks this CTA's contiguous range of (tile, K block) items stage by
// stage with 32-bit counters.  A stage holds g <= G consecutive K blocks of
// one tile; segments (the CTA's blocks of one tile) and fp32 accumulation
// runs (<= RUN_MAX blocks) always end on a stage boundary.
template <int G>
struct Walk {
  int t, kb, kb_first, left, g;
  __device__ Walk(int b0, int b1, int KB) : t(b0 / KB), kb(b0 % KB), kb_first(b0 % KB), left(b1 - b0) { size(KB); }
  __device__ void size(int KB) {
    g = G;
    if (g > left) g = left;
    if (g > KB - kb) g = KB - kb;
  }
  __device__ bool more() const { return left > 0; }
  __device__ bool seg_last(int KB) const { return left == g || kb + g == KB; }
  __device__ bool run_first() const { return ((kb - kb_first) % RUN_MAX) == 0; }
  __device__ bool run_last(int KB) const { return seg_last(KB) || ((kb - kb_first + g) % RUN_MAX) == 0; }
  __device__ void next(int KB) {
    left -= g;
    kb += g;
    if (kb == KB) {
      kb = 0;
      kb_first = 0;
      ++t;
    }
    if (left > 0) size(KB);
  }
};

// Ring position: stage index and the parity of its current phase.
template <int S>
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ void next() {
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Four consecutive K=16 MMAs of one 128-K block (K steps k0..k0+3), issued
// from a single asm statement so that no load can be scheduled between them:
// any memory access by the issuing thread waits until its queued MMAs have
// been accepted by the tensor pipe, which would serialize the burst.
// `acc0` selects accumulate (1) or overwrite (0) for the first MMA only.
template <int NT, int K0>
QUASAR_DEVICE_INLINE void mma_burst4(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t acc0) {
  // B descriptor start advances 32 bytes per K step inside a 64-element swizzle
  // atom and NT*128 bytes per atom (units of 16 bytes in the descriptor).
  constexpr uint64_t o0 = ((K0 + 0) >> 2) * (NT * 8) + ((K0 + 0) & 3) * 2;
  constexpr uint64_t o1 = ((K0 + 1) >> 2) * (NT * 8) + ((K0 + 1) & 3) * 2;
  constexpr uint64_t o2 = ((K0 + 2) >> 2) * (NT * 8) + ((K0 + 2) & 3) * 2;
  constexpr uint64_t o3 = ((K0 + 3) >> 2) * (NT * 8) + ((K0 + 3) & 3) * 2;
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %4, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %4, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %4, t;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem + (K0 + 0) * 8), "l"(bdesc + o0), "r"(acc0), "r"(Cfg<NT>::IDESC),
      "r"(a_tmem + (K0 + 1) * 8), "l"(bdesc + o1), "r"(a_tmem + (K0 + 2) * 8), "l"(bdesc + o2),
      "r"(a_tmem + (K0 + 3) * 8), "l"(bdesc + o3)
      : "memory");
}

template <int NT>
QUASAR_DEVICE_INLINE void drain_acc(uint32_t taddr, int32_t (&acc)[NT / 4]) {
  // NT/4 fp32 accumulator columns, each an exact integer: convert and add.
  uint32_t v[NT / 4];
  if constexpr (NT / 4 == 4) {
    tmem_ld4(taddr, v);
  } else {
#pragma unroll
    for (int g = 0; g < NT / 32; ++g) tmem_ld8(taddr + g * 8, v + g * 8);
  }
  tc_wait_ld();
#pragma unroll
  for (int j = 0; j < NT / 4; ++j) acc[j] += __float2int_rn(__uint_as_float(v[j]));
}

// A finished accumulation run whose TMEM sums still have to be drained, and
// the segment (CTA range within one tile) it closes, if any.
struct PendingRun {
  int R = -1;
  bool flush = false;
  int t = 0, kb_first = 0, kb_last = 0;
  int s2 = 0;        // converted stage holding the run's last blocks
  uint32_t ph2 = 0;  // parity of that stage's MMA-completion phase
};

// Drain run `pr.R` from TMEM into the int32 registers; if it closes a
// segment, publish / finish the segment (see the file comment) and clear the
// registers.  Returns false if a bounded wait ran out.
template <int NT>
QUASAR_DEVICE_INLINE bool finish_run(const PendingRun& pr, int32_t (&acc)[NT / 4], uint64_t* empty2,
                                     uint64_t* accempty, uint32_t tmem_lane, int h, volatile int* abort_flag,
                                     const Params& p, int warp, int lane, int row, int KB, int m_tiles) {
  constexpr int TOK = NT / 4;
  const int a = pr.R & 1;
  // The commit that frees the run's last stage tracks every MMA issued
  // before it, i.e. the whole run: its completion means the sums are final.
  const bool okf = mbar_wait(&empty2[pr.s2], pr.ph2, abort_flag, p.err, SITE_GEMM_ACCFULL, p.limit_ns);
  if (!__all_sync(0xffffffffu, okf)) return false;
  tc_fence_after();
  drain_acc<NT>(tmem_lane + (uint32_t)(a * NT + h * TOK), acc);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&accempty[a]);
  if (!pr.flush) return true;

  const int t = pr.t;
  const int n = (t / m_tiles) * BM + row;
  const int m0 = (t % m_tiles) * NT + h * TOK;
  const bool whole = (pr.kb_first == 0) && (pr.kb_last == KB - 1);
  bool emit = whole;
  if (!whole) {
    // Split tile: publish this warp's 32 x NT/4 sub-tile with integer
    // atomics, then count the K blocks it covered.  The warp that brings the
    // (tile, warp) counter to KB owns the finished sums.
    if (n < p.N) {
#pragma unroll
      for (int jj = 0; jj < TOK; ++jj)
        if (m0 + jj < p.M) atomicAdd(&p.ws_acc[(size_t)(m0 + jj) * p.N + n], acc[jj]);
    }
    __threadfence();
    __syncwarp();
    uint32_t last = 0;
    if (lane == 0) {
      const uint32_t nb = (uint32_t)(pr.kb_last - pr.kb_first + 1);
      const uint32_t old = atomicAdd(&p.ws_cnt[(size_t)t * CONV_WARPS + warp], nb);
      last = (old + nb == (uint32_t)KB) ? 1u : 0u;
    }
    emit = __shfl_sync(0xffffffffu, last, 0) != 0;
    if (emit) {
      __threadfence();
      if (n < p.N) {
#pragma unroll
        for (int jj = 0; jj < TOK; ++jj)
          if (m0 + jj < p.M) acc[jj] = atomicExch(&p.ws_acc[(size_t)(m0 + jj) * p.N + n], 0);
      }
      if (lane == 0) atomicExch(&p.ws_cnt[(size_t)t * CONV_WARPS + warp], 0u);
    }
  }
  if (emit && n < p.N) {
    if (p.acc_out) {
#pragma unroll
      for (int jj = 0; jj < TOK; ++jj)
        if (m0 + jj < p.M) p.acc_out[(size_t)(m0 + jj) * p.N + n] = acc[jj];
    } else {
      const float swn = p.sw[n];
#pragma unroll
      for (int jj = 0; jj < TOK; ++jj) {
        if (m0 + jj < p.M) {
          const float y = __fmul_rn(__fmul_rn(__int2float_rn(acc[jj]), p.sa[m0 + jj]), swn);
          p.Y[(size_t)(m0 + jj) * p.ldy + n] = __float2bfloat16_rn(y);
        }
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < TOK; ++jj) acc[jj] = 0;
  return true;
}

template <int NT, bool XH = false>
__global__ void __launch_bounds__(THREADS, 1)
w8a8_linear_kernel(const __grid_constant__ CUtensorMap tmX, const Params p) {
  using C = Cfg<NT, XH>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage1 = smem;                                  // S1 x [W 16KB | X NT*128]
  uint8_t* b16 = smem + C::S1 * C::STAGE1;                 // S2 x [2 atoms][NT][128B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(b16 + C::S2 * C::B16_BYTES);
  uint64_t* full1 = bars;                     // [S1] copies -> converters
  uint64_t* empty1 = full1 + C::S1;           // [S1] converters -> producer
  uint64_t* full2 = empty1 + C::S1;           // [S2] converters -> MMA
  uint64_t* empty2 = full2 + C::S2;           // [S2] MMA -> converters
  uint64_t* accempty = empty2 + C::S2;        // [2]  drain -> MMA
  uint64_t* mma_done = accempty + 2;          // [1]  final MMA drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Let the next kernel in the stream be scheduled onto SMs as they free up.
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S1; ++s) { mbar_init(&full1[s], 1); mbar_init(&empty1[s], CONV_WARPS); }
    // XH: the producer's fp16 token copy is one more arrival (with its bytes)
    for (int s = 0; s < C::S2; ++s) { mbar_init(&full2[s], CONV_WARPS + (XH ? 1 : 0)); mbar_init(&empty2[s], 1); }
    for (int a = 0; a < 2; ++a) mbar_init(&accempty[a], CONV_WARPS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) prefetch_tmap(&tmX);
  const uint32_t xtx = XH ? (uint32_t)C::B16_BLOCK : 0u;  // bytes of one block's fp16 token tile
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This CTA's contiguous range of (tile, K block) work items.
  const int b0 = (int)((long long)blockIdx.x * p.total / gridDim.x);
  const int b1 = (int)((long long)(blockIdx.x + 1) * p.total / gridDim.x);
  const int KB = p.KB;
  const int m_tiles = p.m_tiles;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      // Weights do not depend on earlier kernels: start streaming the first
      // S1 stages before waiting for the previous kernel.  A stage's blocks
      // are consecutive K blocks of one tile, i.e. contiguous packed bytes.
      int pre = 0;
      {
        Walk<C::G> w(b0, b1, KB);
        for (; pre < C::S1 && w.more(); ++pre, w.next(KB)) {
          mbar_arrive_expect_tx(&full1[pre], (uint32_t)(w.g * (BLOCK_BYTES + C::XB_BYTES)));
          bulk_load(stage1 + pre * C::STAGE1, p.wp + ((size_t)(w.t / m_tiles) * KB + w.kb) * BLOCK_BYTES,
                    (uint32_t)(w.g * BLOCK_BYTES), &full1[pre], pol_w);
        }
      }
      pdl_wait();  // tokens are written by the previous kernel
      Walk<C::G> w(b0, b1, KB);
      Ring<C::S1> rg;
      int issued = 0;
      for (; w.more(); w.next(KB), rg.next(), ++issued) {
        uint8_t* st = stage1 + rg.s * C::STAGE1;
        if (issued >= pre) {
          if (!mbar_wait(&empty1[rg.s], rg.ph ^ 1u, abort_flag, p.err, SITE_GEMM_EMPTY1, p.limit_ns)) break;
          mbar_arrive_expect_tx(&full1[rg.s], (uint32_t)(w.g * (BLOCK_BYTES + C::XB_BYTES)));
          bulk_load(st, p.wp + ((size_t)(w.t / m_tiles) * KB + w.kb) * BLOCK_BYTES, (uint32_t)(w.g * BLOCK_BYTES),
                    &full1[rg.s], pol_w);
        }
        if (!XH)
          for (int b = 0; b < w.g; ++b)
            tma_load_2d(st + C::W_BYTES + b * C::XB_BYTES, &tmX, (w.kb + b) * BK, (w.t % m_tiles) * NT, &full1[rg.s],
                        pol_x);
      }
      // Never leave with copies in flight: wait for the last phase issued on
      // every stage (already complete in a normal run).
      for (int s = 0; s < C::S1 && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / C::S1) * C::S1;
        volatile int dummy = 0;
        mbar_wait(&full1[s], (uint32_t)(last / C::S1) & 1u, &dummy, p.err, SITE_GEMM_DRAIN, p.limit_ns);
      }
    } else if (XH && lane == 1) {
      // fp16 token tiles, straight into the converted ring's B slots (two
      // 64-column swizzle atoms per block), once the MMAs have released them.
      const uint64_t pol_x = policy_evict_last();
      pdl_wait();  // the widened tokens are written by the previous kernel
      Walk<C::G> w(b0, b1, KB);
      Ring<C::S2> r2;
      int issued = 0;
      for (int j = 0; w.more(); ++j, w.next(KB), r2.next(), ++issued) {
        if (j >= C::S2 && !mbar_wait(&empty2[r2.s], r2.ph ^ 1u, abort_flag, p.err, SITE_GEMM_EMPTY2, p.limit_ns))
          break;
        mbar_arrive_expect_tx(&full2[r2.s], (uint32_t)w.g * xtx);
        uint8_t* bd = b16 + r2.s * C::B16_BYTES;
        for (int b = 0; b < w.g; ++b)
          for (int a = 0; a < 2; ++a)
            tma_load_2d(bd + b * C::B16_BLOCK + a * (NT * 128), &tmX, (w.kb + b) * BK + a * 64, (w.t % m_tiles) * NT,
                        &full2[r2.s], pol_x);
      }
      // The MMA warp consumes every phase issued here in a normal run; after
      // an abort, wait (bounded) for the copies of the last phases to land.
      for (int s = 0; s < C::S2 && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / C::S2) * C::S2;
        volatile int dummy = 0;
        mbar_wait(&full2[s], (uint32_t)(last / C::S2) & 1u, &dummy, p.err, SITE_GEMM_DRAIN, p.limit_ns);
      }
    }
  } else if (warp == MMA_WARP || warp == WAITER_WARP) {
    // Any memory access by the thread that issues tcgen05.mma waits until
    // its queued MMAs have been accepted by the tensor pipe, so a barrier
    // wait between stages would drain the pipe.  The waiter warp therefore
    // does every mbarrier wait and releases the MMA warp through a named
    // barrier (no memory access); the reduction over that barrier carries
    // the abort decision, so both warps leave the loop at the same stage and
    // the barrier always completes.
    Walk<C::G> w(b0, b1, KB);
    Ring<C::S2> rg;
    int R = -1;
    const uint64_t bdesc0 = sw128_kmajor_desc(smem_u32(b16));
    for (; w.more(); w.next(KB), rg.next()) {
      const bool run_first = w.run_first();
      if (run_first) ++R;
      uint32_t abort_in = 0;
      if (warp == WAITER_WARP) {
        bool ok = true;
        if (run_first && R >= 2)
          ok = mbar_wait(&accempty[R & 1], ((R >> 1) - 1) & 1, abort_flag, p.err, SITE_GEMM_ACCEMPTY, p.limit_ns);
        ok = ok && mbar_wait(&full2[rg.s], rg.ph, abort_flag, p.err, SITE_GEMM_FULL2, p.limit_ns);
        abort_in = __all_sync(0xffffffffu, ok) ? 0u : 1u;
      }
      if (named_barrier_or(MMA_BAR_ID, 64, abort_in)) break;
      if (warp == MMA_WARP) {
        if (lane == 0) {
          tc_fence_after();
          const uint32_t d_tmem = tmem + (uint32_t)((R & 1) * NT);
          const uint32_t a_tmem = tmem + (uint32_t)(C::TMEM_A0 + rg.s * C::A_COLS);
          const uint64_t bdesc = bdesc0 + (uint64_t)((rg.s * C::B16_BYTES) >> 4);
          const uint32_t acc0 = run_first ? 0u : 1u;
          mma_burst4<NT, 0>(d_tmem, a_tmem, bdesc, acc0);
          mma_burst4<NT, 4>(d_tmem, a_tmem, bdesc, 1u);
          if (w.g == 2) {
            const uint32_t a1 = a_tmem + BK / 2;
            const uint64_t b1 = bdesc + (uint64_t)(C::B16_BLOCK >> 4);
            mma_burst4<NT, 0>(d_tmem, a1, b1, 1u);
            mma_burst4<NT, 4>(d_tmem, a1, b1, 1u);
          }
          tc_commit(&empty2[rg.s]);
        }
        __syncwarp();
      }
    }
    if (warp == MMA_WARP && lane == 0) {
      // Wait until every MMA this thread issued has completed before the CTA
      // may release TMEM.
      tc_commit(mma_done);
      volatile int dummy = 0;
      mbar_wait(mma_done, 0, &dummy, p.err, SITE_GEMM_DRAIN, p.limit_ns);
    }
  } else {
    // ---------------------------------------------------------------- converters
    const int q = warp & 3;       // TMEM lane quadrant = weight rows 32q..32q+31
    const int h = warp >> 2;      // K quarter of each A block; token quarter of the accumulator
    const int row = 32 * q + lane;
    const int ct = threadIdx.x;   // 0..511
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    int32_t acc[C::TOK];
#pragma unroll
    for (int j = 0; j < C::TOK; ++j) acc[j] = 0;

    Walk<C::G> w(b0, b1, KB);
    Ring<C::S1> r1;
    Ring<C::S2> r2;
    int R = -1;
    PendingRun pend;
    for (int j = 0; w.more(); ++j, w.next(KB), r1.next(), r2.next()) {
      const bool run_last = w.run_last(KB);
      const bool seg_last = w.seg_last(KB);
      if (w.run_first()) ++R;

      // Every lane waits; the warp then takes one decision, so the
      // .sync.aligned tcgen05 instructions below always see a full warp.
      bool ok = mbar_wait(&full1[r1.s], r1.ph, abort_flag, p.err, SITE_GEMM_FULL1, p.limit_ns);
      if (j >= C::S2)
        ok = ok && mbar_wait(&empty2[r2.s], r2.ph ^ 1u, abort_flag, p.err, SITE_GEMM_EMPTY2, p.limit_ns);
      if (!__all_sync(0xffffffffu, ok)) break;

      const uint8_t* st = stage1 + r1.s * C::STAGE1;
      // A: this thread's weight row, K quarter h of each block (2 swizzled
      // 16-byte chunks per block).
      for (int b = 0; b < w.g; ++b) {
        uint32_t a[16];
        const uint8_t* wrow = st + b * BLOCK_BYTES + row * 128;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = 2 * h + i;
          const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((c ^ (row & 7)) << 4));
          u8x4_to_f16x4(v.x, a[8 * i + 0], a[8 * i + 1]);   // packed bytes are code + 128
          u8x4_to_f16x4(v.y, a[8 * i + 2], a[8 * i + 3]);
          u8x4_to_f16x4(v.z, a[8 * i + 4], a[8 * i + 5]);
          u8x4_to_f16x4(v.w, a[8 * i + 6], a[8 * i + 7]);
        }
        tmem_st16(tmem + lane_off + (uint32_t)(C::TMEM_A0 + r2.s * C::A_COLS + b * (BK / 2) + 16 * h), a);
      }
      // B: the token tiles, NT rows x 8 chunks per block, widened into the
      // swizzled fp16 tiles (XH: the producer copies them in already widened).
      if (!XH) {
        uint8_t* bd = b16 + r2.s * C::B16_BYTES;
        for (int idx = ct; idx < w.g * NT * 8; idx += CONV_WARPS * 32) {
          const int b = idx / (NT * 8), rem = idx - b * (NT * 8);
          const int xr = rem >> 3, c = rem & 7;
          const uint8_t* xs = st + C::W_BYTES + b * C::XB_BYTES;
          const uint4 v = *reinterpret_cast<const uint4*>(xs + xr * 128 + ((c ^ (xr & 7)) << 4));
          uint4 o0, o1;
          s8x4_to_f16x4(v.x, o0.x, o0.y);
          s8x4_to_f16x4(v.y, o0.z, o0.w);
          s8x4_to_f16x4(v.z, o1.x, o1.y);
          s8x4_to_f16x4(v.w, o1.z, o1.w);
          uint8_t* dst = bd + b * C::B16_BLOCK + (c >> 2) * (NT * 128) + xr * 128;
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
        mbar_arrive(&empty1[r1.s]);
        mbar_arrive(&full2[r2.s]);
      }

      // Drain the run finished one stage ago (its MMAs have had a whole
      // stage to complete), then remember this stage's run if it ends here.
      if (pend.R >= 0) {
        if (!finish_run<NT>(pend, acc, empty2, accempty, tmem + lane_off, h, abort_flag, p, warp, lane, row, KB,
                            m_tiles))
          break;
        pend.R = -1;
      }
      if (run_last) {
        pend.R = R;
        pend.flush = seg_last;
        pend.t = w.t;
        pend.kb_first = w.kb_first;
        pend.kb_last = w.kb + w.g - 1;
        pend.s2 = r2.s;
        pend.ph2 = r2.ph;
      }
    }
    if (pend.R >= 0)
      finish_run<NT>(pend, acc, empty2, accempty, tmem + lane_off, h, abort_flag, p, warp, lane, row, KB, m_tiles);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

// Token tile: the smallest of 16 / 32 / 64 that holds M, else 128 -- or 96
// above 128 tokens when three-quarter tiles pad less (288 = 3 x 96 instead of
// 2 x 128 + a quarter-full third tile).
static int pick_nt(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M > 128 && 96 * ((M + 95) / 96) < 128 * ((M + 127) / 128)) return 96;
  return 128;
}

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

// Token tiles of 96 or 128 on layers of at least 128 weight tiles (N >= 16384):
// the tokens are widened to fp16 once per call (an M x K copy in the
// workspace, one extra launch and a clearing memset) instead of once per
// weight tile inside the kernel.  Measured: gate_up 24576 x 4096 at M = 256
// 95.5 -> 85.3 us; the widening launch costs more than it saves on layers of
// 32-48 tiles (qkv, o_proj, down lose 0.5-2.5 us), so those keep the in-kernel path.
static bool use_xh(int M, const Shape& s) { return !skinny::handles(M) && s.NT >= 96 && s.n_tiles >= 128; }

size_t workspace_size(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  Shape s = shape_of(M, N, K);
  // counters, then the int32 split-K sums of this kernel or the partial-sum
  // slots of the register-path kernel, then (96/128-token tiles) the fp16
  // token copy
  return align256((size_t)s.tiles * CONV_WARPS * 4) +
         align256(std::max((size_t)M * N * 4, skinny::slots_bytes(M, N, K))) +
         (use_xh(M, s) ? align256((size_t)M * K * 2) : 0);
}

// INT8 token codes -> the same values in fp16 (exact), 16 codes per thread.
__global__ void __launch_bounds__(256) widen_tokens_kernel(const int8_t* __restrict__ xq, long long n16,
                                                           uint4* __restrict__ xh) {
  pdl_launch_dependents();
  pdl_wait();  // the codes are written by the previous kernel
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(xq)[i];
    uint4 o0, o1;
    s8x4_to_f16x4(v.x, o0.x, o0.y);
    s8x4_to_f16x4(v.y, o0.z, o0.w);
    s8x4_to_f16x4(v.z, o1.x, o1.y);
    s8x4_to_f16x4(v.w, o1.z, o1.w);
    xh[2 * i] = o0;
    xh[2 * i + 1] = o1;
  }
}

template <int NT, bool XH = false>
static cudaError_t launch_nt(const CUtensorMap& tx, const Params& p, int grid, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(w8a8_linear_kernel<NT, XH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<NT, XH>::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg<NT, XH>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w8a8_linear_kernel<NT, XH>, tx, p);
}

// `xh_ext` (optional, the one-call entry): the token codes already widened to
// fp16 [M][K] by the quantizer; 64- to 128-token tiles then take them from there.
quasar_status_t run(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M, int N, int K,
                    void* Y, int ldy, int32_t* acc_out, void* ws, size_t ws_bytes, cudaStream_t stream,
                    const void* xh_ext = nullptr) {
  if (M < 0 || N <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || N % 8 != 0 || K > 131072) return QUASAR_ERR_UNSUPPORTED;
  if (!acc_out && (ldy < N || ldy % 8 != 0)) return QUASAR_ERR_UNSUPPORTED;
  if (M == 0) return QUASAR_OK;  // empty batch: nothing is read or written
  if (!Xq || !Wp || (!acc_out && (!Y || !sa || !sw))) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(Xq, 16) || !aligned(Wp, 16) || (Y && !aligned(Y, 16)) || (acc_out && !aligned(acc_out, 16)) ||
      (sa && !aligned(sa, 4)) || (sw && !aligned(sw, 4)))
    return QUASAR_ERR_UNSUPPORTED;
  const size_t need = workspace_size(M, N, K);
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return QUASAR_ERR_WORKSPACE;

  Shape s = shape_of(M, N, K);
  uint32_t* ws_cnt = reinterpret_cast<uint32_t*>(ws);
  int32_t* ws_acc = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) + align256((size_t)s.tiles * CONV_WARPS * 4));
  // A few tokens: the register-path kernel (same packed weights, same
  // workspace layout, fewer counters per tile).
  if (skinny::handles(M))
    return skinny::run(Xq, sa, Wp, sw, M, N, K, Y, ldy, acc_out, ws_cnt, ws_acc, stream, false);


  const bool ext = xh_ext != nullptr && s.NT >= 64;
  const bool xh_path = ext || use_xh(M, s);
  uint4* xh = ext ? reinterpret_cast<uint4*>(const_cast<void*>(xh_ext))
              : xh_path ? reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws) +
                                                   align256((size_t)s.tiles * CONV_WARPS * 4) +
                                                   align256(std::max((size_t)M * N * 4, skinny::slots_bytes(M, N, K))))
                        : nullptr;
  CUtensorMap tx;
  if (xh_path) {
    // fp16 copy [M][K]: boxes of 64 values (one 128-byte swizzle row) x NT rows
    if (!encode_2d_bf16(&tx, xh, K, M, K, 64, s.NT)) return QUASAR_ERR_CUDA;
  } else if (!encode_2d_u8(&tx, Xq, K, M, BK, s.NT)) {
    return QUASAR_ERR_CUDA;
  }

  Params p;
  p.wp = reinterpret_cast<const uint8_t*>(Wp);
  p.sa = sa;
  p.sw = sw;
  p.M = M;
  p.N = N;
  p.K = K;
  p.KB = s.KB;
  p.m_tiles = s.m_tiles;
  p.tiles = s.tiles;
  p.total = s.tiles * s.KB;
  p.Y = reinterpret_cast<__nv_bfloat16*>(Y);
  p.ldy = ldy;
  p.acc_out = acc_out;
  p.ws_cnt = ws_cnt;
  p.ws_acc = ws_acc;
  p.err = device_error_word();
  p.limit_ns = wait_limit_ns();
  if (!p.err) return QUASAR_ERR_CUDA;

  const int sms = sm_count();
  if (sms <= 0) return QUASAR_ERR_CUDA;
  const int grid = std::min(p.total, sms);
  cudaError_t e;
  if (xh_path) {
    const long long n16 = (long long)M * K / 16;
    cudaLaunchConfig_t wc = {};
    wc.gridDim = dim3((unsigned)std::min<long long>((n16 + 255) / 256, (long long)sms * 4));
    wc.blockDim = dim3(256);
    wc.stream = stream;
    cudaLaunchAttribute wa[1];
    wa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    wa[0].val.programmaticStreamSerializationAllowed = 1;
    wc.attrs = wa;
    wc.numAttrs = 1;
    e = ext ? cudaSuccess : cudaLaunchKernelEx(&wc, widen_tokens_kernel, Xq, n16, xh);
    if (e == cudaSuccess)
      e = (s.NT == 64)   ? launch_nt<64, true>(tx, p, grid, stream)
          : (s.NT == 96) ? launch_nt<96, true>(tx, p, grid, stream)
                         : launch_nt<128, true>(tx, p, grid, stream);
    // leave the workspace zero-filled (the internal fp16 copy is scratch of this call)
    if (e == cudaSuccess && !ext) e = cudaMemsetAsync(xh, 0, (size_t)M * K * 2, stream);
    return cuda_status(e);
  }
  switch (s.NT) {
    case 16: e = launch_nt<16>(tx, p, grid, stream); break;
    case 32: e = launch_nt<32>(tx, p, grid, stream); break;
    case 64: e = launch_nt<64>(tx, p, grid, stream); break;
    case 96: e = launch_nt<96>(tx, p, grid, stream); break;
    default: e = launch_nt<128>(tx, p, grid, stream); break;
  }
  return cuda_status(e);
}

// ------------------------------------------------------------ 4-bit weights
//
// W4A8: the register-path kernel with 4-bit weight blocks (same schedules,
// same workspace); the token counts it serves (M <= 24) are where the weight
// stream sets the time.
quasar_status_t run_w4(const int8_t* Xq, const float* sa, const int8_t* Wp4, const float* sw, int M, int N, int K,
                       void* Y, int ldy, int32_t* acc_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 0 || N <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || N % 8 != 0 || K > 131072) return QUASAR_ERR_UNSUPPORTED;
  if (!acc_out && (ldy < N || ldy % 8 != 0)) return QUASAR_ERR_UNSUPPORTED;
  if (M == 0) return QUASAR_OK;
  if (!skinny::handles(M)) return QUASAR_ERR_UNSUPPORTED;
  if (!Xq || !Wp4 || (!acc_out && (!Y || !sa || !sw))) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(Xq, 16) || !aligned(Wp4, 16) || (Y && !aligned(Y, 16)) || (acc_out && !aligned(acc_out, 16)) ||
      (sa && !aligned(sa, 4)) || (sw && !aligned(sw, 4)))
    return QUASAR_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < workspace_size(M, N, K) || !aligned(ws, 256)) return QUASAR_ERR_WORKSPACE;
  const Shape s = shape_of(M, N, K);
  uint32_t* ws_cnt = reinterpret_cast<uint32_t*>(ws);
  void* slots = reinterpret_cast<uint8_t*>(ws) + align256((size_t)s.tiles * CONV_WARPS * 4);
  return skinny::run(Xq, sa, Wp4, sw, M, N, K, Y, ldy, acc_out, ws_cnt, slots, stream, true);
}

// ------------------------------------------------------ fused activation path
//
// Smooth + quantize (A2) and the linear (A3 + A4) in one call: the quantizer
// writes codes and scales into the workspace's scratch tail, then the linear
// reads them (two launches, the second overlapping the first through
// programmatic dependent launch).

// The linear's workspace, then the quantizer's codes and scales, then (64- to
// 128-token tiles) the codes again as fp16 for the linear's token operand.
static bool fused_xh(int M, int N, int K) { return !skinny::handles(M) && shape_of(M, N, K).NT >= 64; }

size_t fused_workspace_size(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return workspace_size(M, N, K) + align256((size_t)M * K) + align256((size_t)M * 4) +
         (fused_xh(M, N, K) ? align256((size_t)M * K * 2) : 0);
}

quasar_status_t run_fused(const void* X, int ldx, const float* smooth, const int8_t* Wp, const float* sw, int M,
                          int N, int K, void* Y, int ldy, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 0 || N <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (K % 16 != 0 || N % 8 != 0 || K > 131072) return QUASAR_ERR_UNSUPPORTED;
  if (ldy < N || ldy % 8 != 0 || ldx < K || ldx % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (M == 0) return QUASAR_OK;  // empty batch: nothing is read or written
  if (!X || !smooth || !Wp || !sw || !Y) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(smooth, 16) || !aligned(Wp, 16) || !aligned(Y, 16) || !aligned(sw, 4))
    return QUASAR_ERR_UNSUPPORTED;
  const size_t lin = workspace_size(M, N, K);
  if (!ws || ws_bytes < fused_workspace_size(M, N, K) || !aligned(ws, 256)) return QUASAR_ERR_WORKSPACE;
  int8_t* xq = reinterpret_cast<int8_t*>(ws) + lin;
  float* sa = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + lin + align256((size_t)M * K));
  if (fused_xh(M, N, K)) {
    // The quantizer also writes the codes as fp16: the linear's token
    // operand without a widening launch (rows up to the one-pass kernel's).
    void* xh = reinterpret_cast<uint8_t*>(ws) + lin + align256((size_t)M * K) + align256((size_t)M * 4);
    const quasar_status_t sq = quant::smooth_quant_act_f16(X, ldx, smooth, M, K, xq, sa, xh, stream);
    if (sq == QUASAR_OK) return run(xq, sa, Wp, sw, M, N, K, Y, ldy, nullptr, ws, lin, stream, xh);
    if (sq != QUASAR_ERR_UNSUPPORTED) return sq;
  }
  const quasar_status_t sq = quasar_smooth_quant_act(X, ldx, smooth, M, K, xq, sa, reinterpret_cast<quasar_stream_t>(stream));
  if (sq != QUASAR_OK) return sq;
  return run(xq, sa, Wp, sw, M, N, K, Y, ldy, nullptr, ws, lin, stream);
}

// ---------------------------------------------------------- no-allocation path
//
// For callers that cannot pass a workspace.  The split-K scratch lives in a
// fixed array of this file's device image; host code only ever handles its
// device address, looked up once per device (the symbol itself is a host-side
// stand-in and must never be passed to a kernel).
static __device__ __align__(256) unsigned char g_noalloc_scratch[QUASAR_NOALLOC_SCRATCH_BYTES];

static void* noalloc_scratch_address() {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

quasar_status_t run_noalloc(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M, int N,
                            int K, void* Y, int ldy, cudaStream_t stream) {
  if (M < 0 || N <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (M == 0) return QUASAR_OK;
  const size_t need = workspace_size(M, N, K);
  if (need > QUASAR_NOALLOC_SCRATCH_BYTES) return QUASAR_ERR_WORKSPACE;
  if (!Y) return QUASAR_ERR_INVALID_ARG;
  void* scratch = noalloc_scratch_address();
  if (!scratch) return QUASAR_ERR_CUDA;
  // Start from zeroed counters and sums whatever an earlier call left.
  const cudaError_t e = cudaMemsetAsync(scratch, 0, need, stream);
  if (e != cudaSuccess) return cuda_status(e);
  return run(Xq, sa, Wp, sw, M, N, K, Y, ldy, nullptr, scratch, QUASAR_NOALLOC_SCRATCH_BYTES, stream);
}

}  // namespace gemm
}  // namespace quasar

extern "C" {

quasar_status_t quasar_w8a8_linear_noalloc(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw,
                                           int M, int N, int K, void* Y_bf16, int ldy, quasar_stream_t stream) {
  return quasar::gemm::run_noalloc(Xq, sa, Wp, sw, M, N, K, Y_bf16, ldy, reinterpret_cast<cudaStream_t>(stream));
}

size_t quasar_w8a8_linear_workspace_size(int M, int N, int K) { return quasar::gemm::workspace_size(M, N, K); }

size_t quasar_w8a8_linear_fused_workspace_size(int M, int N, int K) {
  return quasar::gemm::fused_workspace_size(M, N, K);
}

quasar_status_t quasar_w8a8_linear_fused(const void* X_bf16, int ldx, const float* smooth, const int8_t* Wp,
                                         const float* sw, int M, int N, int K, void* Y_bf16, int ldy, void* workspace,
                                         size_t ws_bytes, quasar_stream_t stream) {
  return quasar::gemm::run_fused(X_bf16, ldx, smooth, Wp, sw, M, N, K, Y_bf16, ldy, workspace, ws_bytes,
                                 reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_w8a8_linear(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M,
                                   int N, int K, void* Y_bf16, int ldy, void* workspace, size_t ws_bytes,
                                   quasar_stream_t stream) {
  return quasar::gemm::run(Xq, sa, Wp, sw, M, N, K, Y_bf16, ldy, nullptr, workspace, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_w4a8_linear(const int8_t* Xq, const float* sa, const int8_t* Wp4, const float* sw, int M,
                                   int N, int K, void* Y_bf16, int ldy, void* workspace, size_t ws_bytes,
                                   quasar_stream_t stream) {
  return quasar::gemm::run_w4(Xq, sa, Wp4, sw, M, N, K, Y_bf16, ldy, nullptr, workspace, ws_bytes,
                              reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_int8_gemm_s32(const int8_t* Xq, const int8_t* Wp, int M, int N, int K, int32_t* acc,
                                     void* workspace, size_t ws_bytes, quasar_stream_t stream) {
  if (!acc && M > 0) return QUASAR_ERR_INVALID_ARG;
  return quasar::gemm::run(Xq, nullptr, Wp, nullptr, M, N, K, nullptr, 0, acc, workspace, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
