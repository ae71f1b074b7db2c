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
//  * Swap-AB: weight rows fill the MMA's M = 128 side, tokens the N side:
//    one token tile of up to 256 rows (two of 144 at 257-288 tokens), so each
//    weight block is widened once per launch and meets every token in one
//    instruction per K step.  A kind::f16 MMA of M = 128, K = 16 costs ~114
//    cycles for any N <= 192 and ~138 at N = 256 (measured with
//    quasar_probe_tensor_rate), so at a few tokens this kernel is bound by 8
//    such instructions per 16 KB weight block, not by its operands.
//  * The weight tile is the A operand and lives in TMEM: converter warps read
//    the INT8 tile from shared memory, widen it in registers and tcgen05.st
//    it into TMEM.  The token tile is the B operand in a 128B-swizzled
//    K-major shared-memory layout, widened in the kernel for tiles of up to
//    64 rows, or copied in already widened (an fp16 copy made once per call)
//    by TMA for wider tiles.
//  * Weights arrive pre-packed (quasar_pack_weights) as contiguous 16 KB
//    blocks of 128 rows x 128 K, rows already in the 128B-swizzled order and
//    each code stored biased by +128, so one 1-D bulk copy per block streams
//    them from HBM and widening a byte takes no sign fix-up.  The W4A8
//    variant streams 8 KB blocks of 4-bit codes (quasar_pack_weights_w4) and
//    widens nibbles instead; the rest of the kernel is the same.
//  * Work split, chosen per shape by a cost in blocks (split_of): a cluster
//    of 2-4 CTAs per weight tile, each a K part, the parts pushed into the
//    CTA that finishes each row slice through distributed shared memory; K
//    parts per tile summed with integer atomics into a zero-filled workspace
//    (completion counted per (tile, converter warp): the warp that completes
//    a sub-tile applies the epilogue and re-zeroes what it used; no CTA ever
//    waits on another); whole tiles; or equal contiguous ranges of the
//    (tile, K block) list over one CTA per SM (stream-K).
//  * Programmatic dependent launch: the weight stream of the first stages
//    starts before the previous kernel in the stream has finished; token
//    loads and every global write wait for it (griddepcontrol.wait).
//  * Warp roles: warps 0-15 convert (and drain / run the epilogue), warp 16
//    issues the copies, warp 17 issues MMAs, warp 18 does every mbarrier
//    wait for the MMA warp; tiles of >= 128 rows add a spare warp so that the
//    fifth warpgroup can hand registers to the converters (setmaxnreg).
#include <algorithm>
#include <mutex>

#include "quasar_common.cuh"

namespace quasar {
namespace skinny {  // w8a8_skinny.cu: the register-path kernel, a few tokens (skinny::handles)
struct FusedIn {
  const void* X;
  int ldx;
  const float* smooth;
};
bool handles(int M, int N);
size_t slots_bytes(int M, int N, int K);
quasar_status_t run(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M, int N, int K,
                    void* Y, int ldy, int32_t* acc_out, uint32_t* ws_cnt, void* slots, cudaStream_t stream,
                    bool w4, const FusedIn* fin);
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
constexpr int MMA_BAR_ID = 1;   // named barrier pairing the MMA and waiter warps
constexpr int CONV_BAR_ID = 2;  // named barrier of the converter warps
constexpr int TMEM_COLS = 512;
constexpr int BLOCK_BYTES = BM * BK;   // one packed weight block
constexpr int SMEM_OPTIN = 232448;     // shared memory a block may opt into

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A/B fp16
// (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
template <int NT>
__host__ __device__ constexpr uint32_t idesc() {
  return (1u << 4) | (uint32_t(NT >> 3) << 17) | (uint32_t(BM >> 4) << 24);
}

// NT: token rows of one tile (the MMA's N).  XH: the token codes arrive
// already widened to fp16 (one copy per call in the workspace, or written by
// the quantizer of the one-call entry) and are copied by TMA straight into
// the MMA's B layout; the converters then widen only the weights, and the
// INT8 ring carries weight blocks alone.  W4: the weights arrive as 4-bit
// blocks (quasar_pack_weights_w4: 8 KB per 128 x 128 block) and are widened
// from nibbles; everything after the widening is the INT8 kernel's.
template <int NT, bool XH = false, bool W4 = false>
struct Cfg {
  // Wide tiles (NT >= 128) keep NT/4 int32 run sums per converter thread.
  // A fifth warpgroup (copy, MMA, waiter and one spare warp) lets the block
  // move registers from those warps to the converters (setmaxnreg): launched
  // at REGS_LAUNCH per thread, the converters rise to REGS_CONV and the
  // fifth warpgroup drops to REGS_AUX, which gives back exactly what the
  // converters take.  The host checks the launch count before using it.
  static constexpr bool WIDE = NT >= 128;
  static constexpr int WARPS = CONV_WARPS + (WIDE ? 4 : 3);
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int REGS_LAUNCH = 96;
  static constexpr int REGS_CONV = NT >= 192 ? 112 : 104;
  static constexpr int REGS_AUX = NT >= 192 ? 32 : 64;
  // Blocks per pipeline stage: two 128-K blocks per handshake halve the
  // per-byte cost of the barrier round trips; NT >= 96 keeps one (TMEM).
  static constexpr int G = (NT >= 96) ? 1 : 2;
  static constexpr int A_COLS = G * BK / 2;                  // TMEM columns per A stage (fp16 pairs)
  // Accumulators in TMEM: two (a run drains while the next accumulates)
  // unless the tile is too wide to leave room for the A stages.
  static constexpr int NACC = (2 * NT + 2 * A_COLS <= TMEM_COLS) ? 2 : 1;
  static constexpr int TMEM_A0 = NACC * NT;                  // A stages follow the accumulators
  // Converted stages (TMEM A + shared-memory B) and INT8 stages, sized so
  // that the operand bytes in flight cover the copy latency at each width.
  static constexpr int S2 = XH ? (NT == 256 ? 3 : NT == 192 ? 2 : NT == 144 ? 3 : NT == 128 ? 4 : 2)
                               : (NT == 64 ? 2 : 3);
  static constexpr int WBLK = W4 ? BLOCK_BYTES / 2 : BLOCK_BYTES;   // bytes of one packed weight block
  static constexpr int W_BYTES = G * WBLK;                   // weight blocks of a stage
  static constexpr int XB_BYTES = XH ? 0 : NT * BK;          // INT8 token tile of one block
  static constexpr int STAGE1 = W_BYTES + G * XB_BYTES;      // multiple of 1024
  static constexpr int B16_BLOCK = NT * BK * 2;              // fp16 token tile of one block (2 atoms)
  static constexpr int B16_BYTES = G * B16_BLOCK;
  static constexpr int S1_FIT = (SMEM_OPTIN - 1024 - 256 - S2 * B16_BYTES) / STAGE1;
  // (4-bit blocks: as many stages as fit, up to 8, for the same bytes in flight)
  static constexpr int S1 = (XH || W4) ? (S1_FIT < 8 ? S1_FIT : 8) : (NT == 16) ? 5 : (NT == 32) ? 4 : 3;
  static constexpr int TOK = NT / 4;                         // accumulator columns per converter thread
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + S1 * STAGE1 + S2 * B16_BYTES + BAR_BYTES;
  static_assert(RUN_MAX % G == 0, "stages never straddle an accumulation run");
  static_assert(TMEM_A0 + S2 * A_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(STAGE1 % 1024 == 0 && B16_BLOCK % 1024 == 0, "1024B alignment of swizzled tiles");
  static_assert(S1 >= 2 && S2 >= 2, "pipeline depth");
  // The partial sums a CTA of a cluster receives (csize senders x NT columns
  // x its share of the rows: at most 132 rows' worth, 3 x 44) go over the
  // INT8 ring and the epilogue scales over the converted ring (both idle by
  // then), or the other way round when the converted ring is the one that
  // holds the sums; where neither does (4-bit blocks at 192-row tiles) the
  // sums span both rings, which are contiguous, and the scales take the
  // converted ring's last KB.  Offsets from the start of the INT8 ring.
  static constexpr int PART_BYTES = 132 * NT * 4;
  static constexpr int SC_BYTES = (BM + NT) * 4;
  static constexpr int PART_MODE = PART_BYTES <= S1 * STAGE1 ? 0 : PART_BYTES <= S2 * B16_BYTES ? 1 : 2;
  static constexpr int PART_OFF = PART_MODE == 1 ? S1 * STAGE1 : 0;
  static constexpr int SC_OFF = PART_MODE == 0 ? S1 * STAGE1
                                : PART_MODE == 1 ? 0
                                                 : S1 * STAGE1 + S2 * B16_BYTES - ((SC_BYTES + 1023) & ~1023);
  static_assert(PART_MODE != 2 || PART_BYTES <= SC_OFF, "cluster partial sums fit");
  static_assert(SC_BYTES <= (PART_MODE == 0 ? S2 * B16_BYTES : PART_MODE == 1 ? S1 * STAGE1 : SC_BYTES),
                "epilogue scales fit");
  static_assert(SMEM <= SMEM_OPTIN, "shared memory budget");
  static_assert(NT % 16 == 0 && NT <= 256 && TOK % 4 == 0, "MMA N");
  static_assert(!WIDE || XH, "wide tiles take the fp16 token copy");
  static_assert(!WIDE || (CONV_WARPS * 32 * (REGS_CONV - REGS_LAUNCH) <= 4 * 32 * (REGS_LAUNCH - REGS_AUX)),
                "register split: the converters never take more than the fifth warpgroup returns");
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
  int tile_ranges; // 1: each CTA takes whole tiles (a contiguous run of them), never part of one
  int csize;       // > 1: thread-block clusters of csize CTAs, one per tile, each CTA a K part;
                   // the parts are summed through distributed shared memory
  int pre;         // weight stages issued before waiting for the previous kernel
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
      ::"r"(d_tmem), "r"(a_tmem + (K0 + 0) * 8), "l"(bdesc + o0), "r"(acc0), "r"(idesc<NT>()),
      "r"(a_tmem + (K0 + 1) * 8), "l"(bdesc + o1), "r"(a_tmem + (K0 + 2) * 8), "l"(bdesc + o2),
      "r"(a_tmem + (K0 + 3) * 8), "l"(bdesc + o3)
      : "memory");
}

// TOK fp32 accumulator columns of this thread's TMEM lane, each an exact
// integer: convert and add to the int32 run sums, 16 columns per load (then
// 8 and 4 for the tail) so that the temporaries stay small next to the sums
// (measured: two loads per wait spilled at wide tiles and ran slower).
template <int TOK>
QUASAR_DEVICE_INLINE void drain_acc(uint32_t taddr, int32_t (&acc)[TOK]) {
#pragma unroll
  for (int c = 0; c + 16 <= TOK; c += 16) {
    uint32_t v[16];
    tmem_ld16(taddr + c, v);
    tc_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[c + j] += __float2int_rn(__uint_as_float(v[j]));
  }
  constexpr int T1 = TOK & ~15;
  if constexpr ((TOK & 8) != 0) {
    uint32_t v[8];
    tmem_ld8(taddr + T1, v);
    tc_wait_ld();
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[T1 + j] += __float2int_rn(__uint_as_float(v[j]));
  }
  constexpr int T2 = TOK & ~7;
  if constexpr ((TOK & 4) != 0) {
    uint32_t v[4];
    tmem_ld4(taddr + T2, v);
    tc_wait_ld();
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[T2 + j] += __float2int_rn(__uint_as_float(v[j]));
  }
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
template <int NT, int NACC>
QUASAR_DEVICE_INLINE bool finish_run(const PendingRun& pr, int32_t (&acc)[NT / 4], uint64_t* empty2,
                                     uint64_t* accempty, uint32_t tmem_lane, int h, volatile int* abort_flag,
                                     const Params& p, int warp, int lane, int row, int KB, int m_tiles) {
  constexpr int TOK = NT / 4;
  const int a = pr.R % NACC;
  // The commit that frees the run's last stage tracks every MMA issued
  // before it, i.e. the whole run: its completion means the sums are final.
  const bool okf = mbar_wait(&empty2[pr.s2], pr.ph2, abort_flag, p.err, SITE_GEMM_ACCFULL, p.limit_ns);
  if (!__all_sync(0xffffffffu, okf)) return false;
  tc_fence_after();
  drain_acc<TOK>(tmem_lane + (uint32_t)(a * NT + h * TOK), acc);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&accempty[a]);
  if (!pr.flush) return true;
  if (p.csize > 1) return true;   // summed across the cluster after the loop

  const int t = pr.t;
  const int n = (t / m_tiles) * BM + row;
  const int m0 = (t % m_tiles) * NT + h * TOK;
  const bool whole = (pr.kb_first == 0) && (pr.kb_last == KB - 1);
  bool emit = whole;
  // The row's channel scale, loaded now so that its latency overlaps the
  // publication below instead of following it.
  const float swn = (!p.acc_out && n < p.N) ? __ldg(p.sw + n) : 0.f;
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
      // acquire-release: the warp that completes the count sees every other
      // contributor's sums (each fenced before its count)
      const uint32_t nb = (uint32_t)(pr.kb_last - pr.kb_first + 1);
      uint32_t old;
      asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;"
                   : "=r"(old)
                   : "l"(&p.ws_cnt[(size_t)t * CONV_WARPS + warp]), "r"(nb)
                   : "memory");
      last = (old + nb == (uint32_t)KB) ? 1u : 0u;
    }
    emit = __shfl_sync(0xffffffffu, last, 0) != 0;
    if (emit) {
      // Every contribution is in L2 now (lane 0's acquire, shared with the
      // warp by the barrier): take the sums and leave zeros for the next
      // call in one atomic exchange each (measured faster than plain loads
      // followed by plain stores).
      __syncwarp();
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
#pragma unroll
      for (int jj = 0; jj < TOK; ++jj) {
        if (m0 + jj < p.M) {
          const float y = __fmul_rn(__fmul_rn(__int2float_rn(acc[jj]), __ldg(p.sa + m0 + jj)), swn);
          p.Y[(size_t)(m0 + jj) * p.ldy + n] = __float2bfloat16_rn(y);
        }
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < TOK; ++jj) acc[jj] = 0;
  return true;
}



// Cluster phase of a split tile (csize CTAs, one K part each).  CTA `rank`
// finishes the rows [4 u0, 4 u1) of the tile (units of four rows split evenly
// over the cluster).  Every CTA first pushes its int32 sums for those rows
// into that CTA's shared memory (remote stores, which the sender does not
// wait for; measured, pulling them with remote loads ran at ~30 GB/s per
// SM), laid out [sender rank][token column][row - 4 u0] with a row stride of
// rows_per_rank(csize) (at most 64, for a cluster of 2); after a release /
// acquire cluster barrier each CTA adds the csize parts from its own shared
// memory and writes its rows (dequantized, or the int32 sums).  Four
// consecutive rows per item: consecutive threads on consecutive rows of Y.

QUASAR_DEVICE_INLINE int rows_per_rank(int csize) { return (((BM / 4) + csize - 1) / csize) * 4; }
QUASAR_DEVICE_INLINE int rank_first_unit(int r, int csize) { return r * (BM / 4) / csize; }

QUASAR_DEVICE_INLINE void st_cluster_u32(uint32_t remote_addr, int32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote_addr), "r"(v) : "memory");
}


// This thread's TOK sums (weight row `row`, token columns h*TOK ..) pushed
// to the CTA that finishes the row.
template <int NT>
QUASAR_DEVICE_INLINE void cluster_push(const Params& p, int32_t* part, const int32_t (&acc)[NT / 4], int row, int h,
                                       int my_rank) {
  constexpr int TOK = NT / 4;
  const int csize = p.csize;
  const int rpr = rows_per_rank(csize);
  int owner = 0;
  while (owner + 1 < csize && rank_first_unit(owner + 1, csize) * 4 <= row) ++owner;
  const int lr = row - rank_first_unit(owner, csize) * 4;
  const uint32_t base = map_to_rank(part, (uint32_t)owner);
  const uint32_t at = base + (uint32_t)(((my_rank * NT + h * TOK) * rpr + lr) * 4);
#pragma unroll
  for (int jj = 0; jj < TOK; ++jj) st_cluster_u32(at + (uint32_t)(jj * rpr * 4), acc[jj]);
}

// The epilogue scales of tile t in shared memory (sw of its 128 weight rows,
// then sa of its NT token rows), loaded ahead so that the finalize reads
// no global memory.
template <int NT>
QUASAR_DEVICE_INLINE void stage_scales(const Params& p, float* sc, int t, int ct) {
  const int n_base = (t / p.m_tiles) * BM;
  const int m_base = (t % p.m_tiles) * NT;
  if (p.acc_out) return;
  for (int i = ct; i < BM + NT; i += CONV_WARPS * 32) {
    if (i < BM) {
      sc[i] = n_base + i < p.N ? __ldg(p.sw + n_base + i) : 0.f;
    } else {
      const int m = m_base + (i - BM);
      sc[i] = m < p.M ? __ldg(p.sa + m) : 0.f;
    }
  }
}

template <int NT>
QUASAR_DEVICE_INLINE void cluster_finalize(const Params& p, const int32_t* part, const float* sc, int t, int rank,
                                           int ct) {
  const int csize = p.csize;   // 2 .. 4
  const int rpr = rows_per_rank(csize);
  const int u0 = rank_first_unit(rank, csize), u1 = rank_first_unit(rank + 1, csize);
  const int nu = u1 - u0;
  const int n_base = (t / p.m_tiles) * BM;
  const int m_base = (t % p.m_tiles) * NT;
  for (int i = ct; i < nu * NT; i += CONV_WARPS * 32) {
    const int col = i / nu, lu = i - col * nu;
    const int m = m_base + col;
    const int n = n_base + 4 * (u0 + lu);
    if (m >= p.M || n >= p.N) continue;
    int4 v = make_int4(0, 0, 0, 0);
    for (int q = 0; q < csize; ++q) {
      const int4 x = *reinterpret_cast<const int4*>(part + (q * NT + col) * rpr + 4 * lu);
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    if (p.acc_out) {
      *reinterpret_cast<int4*>(p.acc_out + (size_t)m * p.N + n) = v;
    } else {
      const float sam = sc[BM + col];
      const float4 swv = *reinterpret_cast<const float4*>(sc + n - n_base);
      const float y0 = __fmul_rn(__fmul_rn(__int2float_rn(v.x), sam), swv.x);
      const float y1 = __fmul_rn(__fmul_rn(__int2float_rn(v.y), sam), swv.y);
      const float y2 = __fmul_rn(__fmul_rn(__int2float_rn(v.z), sam), swv.z);
      const float y3 = __fmul_rn(__fmul_rn(__int2float_rn(v.w), sam), swv.w);
      const __nv_bfloat162 lo = __halves2bfloat162(__float2bfloat16_rn(y0), __float2bfloat16_rn(y1));
      const __nv_bfloat162 hi = __halves2bfloat162(__float2bfloat16_rn(y2), __float2bfloat16_rn(y3));
      uint2 out;
      out.x = *reinterpret_cast<const uint32_t*>(&lo);
      out.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(p.Y + (size_t)m * p.ldy + n) = out;
    }
  }
}

// Which warp roles one copy of the kernel body contains: all of them, or
// (wide tiles, after the register split) the converters or the other warps
// alone, so that each copy is compiled under its own register limit.
enum Roles { ROLES_ALL = 0, ROLES_CONV = 1, ROLES_AUX = 2 };

template <int NT, bool XH, bool W4, int ROLES>
QUASAR_DEVICE_INLINE void linear_body(const CUtensorMap& tmX, const Params& p) {
  using C = Cfg<NT, XH, W4>;
  constexpr bool CONV = ROLES != ROLES_AUX;   // this copy runs the converter warps
  constexpr bool AUX = ROLES != ROLES_CONV;   // this copy runs the copy / MMA / waiter warps
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage1 = smem;                                  // S1 x [W G x WBLK | X G x NT*128]
  uint8_t* b16 = smem + C::S1 * C::STAGE1;                 // S2 x [2 atoms][NT][128B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(b16 + C::S2 * C::B16_BYTES);
  uint64_t* full1 = bars;                     // [S1] copies -> converters
  uint64_t* empty1 = full1 + C::S1;           // [S1] converters -> producer
  uint64_t* full2 = empty1 + C::S1;           // [S2] converters -> MMA
  uint64_t* empty2 = full2 + C::S2;           // [S2] MMA -> converters
  uint64_t* accempty = empty2 + C::S2;        // [NACC] drain -> MMA
  uint64_t* mma_done = accempty + 2;          // [1]  final MMA drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Let the next kernel in the stream be scheduled onto SMs as they free up.
  pdl_launch_dependents();

  if (CONV && threadIdx.x == 0) {
    for (int s = 0; s < C::S1; ++s) { mbar_init(&full1[s], 1); mbar_init(&empty1[s], CONV_WARPS); }
    // XH: the producer's fp16 token copy is one more arrival (with its bytes)
    for (int s = 0; s < C::S2; ++s) { mbar_init(&full2[s], CONV_WARPS + (XH ? 1 : 0)); mbar_init(&empty2[s], 1); }
    for (int a = 0; a < C::NACC; ++a) mbar_init(&accempty[a], CONV_WARPS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (AUX && warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (AUX && warp == PRODUCER_WARP && lane == 0) prefetch_tmap(&tmX);
  const uint32_t xtx = XH ? (uint32_t)C::B16_BLOCK : 0u;  // bytes of one block's fp16 token tile
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This CTA's contiguous range of (tile, K block) work items.
  const int b0 = p.tile_ranges ? (int)((long long)blockIdx.x * p.tiles / gridDim.x) * p.KB
                               : (int)((long long)blockIdx.x * p.total / gridDim.x);
  const int b1 = p.tile_ranges ? (int)((long long)(blockIdx.x + 1) * p.tiles / gridDim.x) * p.KB
                               : (int)((long long)(blockIdx.x + 1) * p.total / gridDim.x);
  const int KB = p.KB;
  const int m_tiles = p.m_tiles;

  if (AUX && warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      // Weights do not depend on earlier kernels: start streaming the first
      // p.pre stages before waiting for the previous kernel (the host picks
      // the depth).  A stage's blocks are consecutive K blocks of one tile,
      // i.e. contiguous packed bytes.
      int pre = 0;
      {
        Walk<C::G> w(b0, b1, KB);
        for (; pre < C::S1 && pre < p.pre && w.more(); ++pre, w.next(KB)) {
          mbar_arrive_expect_tx(&full1[pre], (uint32_t)(w.g * (C::WBLK + C::XB_BYTES)));
          bulk_load(stage1 + pre * C::STAGE1, p.wp + ((size_t)(w.t / m_tiles) * KB + w.kb) * C::WBLK,
                    (uint32_t)(w.g * C::WBLK), &full1[pre], pol_w);
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
          mbar_arrive_expect_tx(&full1[rg.s], (uint32_t)(w.g * (C::WBLK + C::XB_BYTES)));
          bulk_load(st, p.wp + ((size_t)(w.t / m_tiles) * KB + w.kb) * C::WBLK, (uint32_t)(w.g * C::WBLK),
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
    __syncwarp();
    if (p.csize > 1) {   // the converters' two cluster barriers (no data of this warp crosses them)
      cluster_sync_exec();
      cluster_sync_exec();
    }
  } else if (AUX && (warp == MMA_WARP || warp == WAITER_WARP)) {
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
        if (run_first && R >= C::NACC)
          ok = mbar_wait(&accempty[R % C::NACC], (uint32_t)((R / C::NACC) - 1) & 1u, abort_flag, p.err,
                         SITE_GEMM_ACCEMPTY, p.limit_ns);
        ok = ok && mbar_wait(&full2[rg.s], rg.ph, abort_flag, p.err, SITE_GEMM_FULL2, p.limit_ns);
        abort_in = __all_sync(0xffffffffu, ok) ? 0u : 1u;
      }
      if (named_barrier_or(MMA_BAR_ID, 64, abort_in)) break;
      if (warp == MMA_WARP) {
        if (lane == 0) {
          tc_fence_after();
          const uint32_t d_tmem = tmem + (uint32_t)((R % C::NACC) * NT);
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
    __syncwarp();
    if (p.csize > 1) {   // the converters' two cluster barriers (no data of this warp crosses them)
      cluster_sync_exec();
      cluster_sync_exec();
    }
  } else if (CONV && warp < CONV_WARPS) {
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
      // 16-byte chunks per block; 4-bit blocks: one chunk, 64-byte rows).
      for (int b = 0; b < w.g; ++b) {
        uint32_t a[16];
        if constexpr (W4) {
          // Byte 4 i + j holds code(32 h + 4 i + j) + 8 in its low nibble and
          // code(32 h + 16 + 4 i + j) + 8 in its high nibble.
          const uint4 v = *reinterpret_cast<const uint4*>(st + b * C::WBLK + row * 64 + ((h ^ ((row >> 1) & 3)) << 4));
          const uint32_t d[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            n4x4_to_f16x4(d[i] & 0x0F0F0F0Fu, a[2 * i], a[2 * i + 1]);
            n4x4_to_f16x4((d[i] >> 4) & 0x0F0F0F0Fu, a[8 + 2 * i], a[9 + 2 * i]);
          }
        } else {
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
        if (!finish_run<NT, C::NACC>(pend, acc, empty2, accempty, tmem + lane_off, h, abort_flag, p, warp, lane,
                                     row, KB, m_tiles))
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
      finish_run<NT, C::NACC>(pend, acc, empty2, accempty, tmem + lane_off, h, abort_flag, p, warp, lane, row, KB,
                              m_tiles);
    __syncwarp();
    if (p.csize > 1) {
      // Split tile of a cluster: the sums go to the CTA that finishes their
      // rows, into its rings, which the first barrier shows idle in every
      // CTA (all blocks converted, every MMA complete).
      int32_t* part = reinterpret_cast<int32_t*>(stage1 + C::PART_OFF);
      float* sc = reinterpret_cast<float*>(stage1 + C::SC_OFF);
      const int my_rank = (int)(blockIdx.x % (unsigned)p.csize);
      named_barrier_or(CONV_BAR_ID, CONV_WARPS * 32, 0u);   // every converter is past the rings
      stage_scales<NT>(p, sc, b0 / KB, ct);
      cluster_sync_exec();
      cluster_push<NT>(p, part, acc, row, h, my_rank);
      cluster_sync_full();
      cluster_finalize<NT>(p, part, sc, b0 / KB, my_rank, ct);
    }
  } else if (p.csize > 1) {
    // the spare warp of the fifth warpgroup
    cluster_sync_exec();
    cluster_sync_exec();
  }

  tc_fence_before();
  __syncthreads();
  if (AUX && warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int NT, bool XH = false, bool W4 = false>
__global__ void __launch_bounds__(Cfg<NT, XH, W4>::THREADS, 1)
w8a8_linear_kernel(const __grid_constant__ CUtensorMap tmX, const Params p) {
  using C = Cfg<NT, XH, W4>;
  if constexpr (C::WIDE) {
    // Move registers from the fifth warpgroup to the converters before
    // anything else runs (warpgroup-uniform: warps 0-15 and 16-19); each
    // side then runs its own copy of the body under its own limit.
    if ((threadIdx.x >> 5) < CONV_WARPS) {
      regs_inc<C::REGS_CONV>();
      linear_body<NT, XH, W4, ROLES_CONV>(tmX, p);
    } else {
      regs_dec<C::REGS_AUX>();
      linear_body<NT, XH, W4, ROLES_AUX>(tmX, p);
    }
  } else {
    linear_body<NT, XH, W4, ROLES_ALL>(tmX, p);
  }
}

// ------------------------------------------------------------------ host side

// Token tile: the smallest of 16 / 32 / 64 / 128 / 144 / 192 / 256 rows that
// holds M, so that every weight block is widened once per launch and meets
// all tokens in one accumulator.  Measured (quasar_probe_tensor_rate): a
// kind::f16 MMA of M = 128, K = 16 costs ~114 cycles for every N <= 192 and
// ~138 at N = 256, so one wide tile beats two narrow passes (256 tokens:
// 8 x 138 cycles per weight block instead of 16 x 114).  257-288 tokens (32
// sequences x 9 positions) need two instructions per K step whatever the
// split: two 144-row tiles; more tokens, 256-row tiles.
static int pick_nt(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  if (M <= 144) return 144;
  if (M <= 192) return 192;
  if (M <= 256) return 256;
  if (M <= 288) return 144;
  return 256;
}

struct Shape {
  int NT, m_tiles, n_tiles, tiles, KB;
};

static Shape shape_with(int M, int N, int K, int nt) {
  Shape s;
  s.NT = nt;
  s.m_tiles = (M + s.NT - 1) / s.NT;
  s.n_tiles = (N + BM - 1) / BM;
  s.tiles = s.n_tiles * s.m_tiles;
  s.KB = (K + BK - 1) / BK;
  return s;
}

static Shape shape_of(int M, int N, int K) { return shape_with(M, N, K, pick_nt(M)); }

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Tiles of 128 rows and more always take the fp16 token copy: widening the
// tokens inside the kernel would cost the converters more than the weights
// per block.  Through quasar_w8a8_linear the copy is made by one small
// launch into the workspace (and cleared afterwards); the one-call entry's
// quantizer writes it directly.
static bool use_xh(int M, int N, const Shape& s) { return !skinny::handles(M, N) && s.NT >= 128; }

// Counter region: one counter per (tile, converter warp), sized for the
// 64-row fallback of wide tiles too so that both use the same layout.
static size_t cnt_bytes(int M, int N, int K) {
  const Shape s = shape_of(M, N, K);
  const int tiles = std::max(s.tiles, shape_with(M, N, K, std::min(s.NT, 64)).tiles);
  return align256((size_t)tiles * CONV_WARPS * 4);
}

// The prefix that must be zero when a call starts: the counters and, on the
// tcgen05 path, the int32 sums of split tiles.  The register-path kernel's
// partial-sum slots and the fp16 token copy need no initial content.
size_t zeroed_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return cnt_bytes(M, N, K) + (skinny::handles(M, N) ? 0 : align256((size_t)M * N * 4));
}

size_t workspace_size(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  Shape s = shape_of(M, N, K);
  // counters, then the int32 split-K sums of this kernel or the partial-sum
  // slots of the register-path kernel, then (tiles of >= 128 rows) the fp16
  // token copy
  return cnt_bytes(M, N, K) + align256(std::max((size_t)M * N * 4, skinny::slots_bytes(M, N, K))) +
         (use_xh(M, N, s) ? align256((size_t)M * K * 2) : 0);
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

// Wide variants rely on the block's register split: the launch count must
// leave the converters' increase covered by what the fifth warpgroup gives
// back.  Checked once per device against the compiled kernel; 0 = usable.
template <int NT, bool XH, bool W4>
static cudaError_t check_split(int dev) {
  using C = Cfg<NT, XH, W4>;
  if constexpr (!C::WIDE) {
    return cudaSuccess;
  } else {
    static int state[64] = {0};   // 0 unknown, 1 usable, 2 not usable
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!state[dev]) {
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, w8a8_linear_kernel<NT, XH, W4>);
      if (e != cudaSuccess) return e;
      const int r = fa.numRegs;
      const bool ok = r >= C::REGS_AUX && r <= C::REGS_CONV &&
                      (long long)CONV_WARPS * 32 * (C::REGS_CONV - r) <= (long long)4 * 32 * (r - C::REGS_AUX);
      state[dev] = ok ? 1 : 2;
    }
    return state[dev] == 1 ? cudaSuccess : cudaErrorNotSupported;
  }
}

template <int NT, bool XH, bool W4>
static cudaError_t configure(int dev) {
  static int configured[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(w8a8_linear_kernel<NT, XH, W4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<NT, XH, W4>::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return check_split<NT, XH, W4>(dev);
}

template <int NT, bool XH, bool W4>
static cudaLaunchConfig_t config_of(int grid, int csize, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg<NT, XH, W4>::THREADS);
  cfg.dynamicSmemBytes = Cfg<NT, XH, W4>::SMEM;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)csize;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = csize > 1 ? 2 : 1;
  return cfg;
}

// Clusters of `csize` CTAs of this variant the device keeps resident at once
// (0 if unknown); cached per device and size.
template <int NT, bool XH, bool W4>
static int resident_clusters(int dev, int csize) {
  static int cache[64][5];
  static bool init[64][5] = {};
  if (dev < 0 || dev >= 64 || csize < 2 || csize > 4) return 0;
  if (!init[dev][csize]) {
    int n = 0;
    if (configure<NT, XH, W4>(dev) == cudaSuccess) {
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = config_of<NT, XH, W4>(csize * 8, csize, nullptr, attr);
      if (cudaOccupancyMaxActiveClusters(&n, w8a8_linear_kernel<NT, XH, W4>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache[dev][csize] = n;
    init[dev][csize] = true;
  }
  return cache[dev][csize];
}

template <int NT, bool XH, bool W4>
static cudaError_t launch_nt(const CUtensorMap& tx, const Params& p, int grid, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = configure<NT, XH, W4>(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = config_of<NT, XH, W4>(grid, p.csize, stream, attr);
  return cudaLaunchKernelEx(&cfg, w8a8_linear_kernel<NT, XH, W4>, tx, p);
}

// The variant for a tile width: fp16 token copy (xh) or in-kernel widening.
template <bool W4>
static cudaError_t launch_tc(int nt, bool xh, const CUtensorMap& tx, const Params& p, int grid, cudaStream_t stream) {
  if (xh) {
    switch (nt) {
      case 64: return launch_nt<64, true, W4>(tx, p, grid, stream);
      case 128: return launch_nt<128, true, W4>(tx, p, grid, stream);
      case 144: return launch_nt<144, true, W4>(tx, p, grid, stream);
      case 192: return launch_nt<192, true, W4>(tx, p, grid, stream);
      default: return launch_nt<256, true, W4>(tx, p, grid, stream);
    }
  }
  switch (nt) {   // tiles of >= 128 rows always take the fp16 copy
    case 16: return launch_nt<16, false, W4>(tx, p, grid, stream);
    case 32: return launch_nt<32, false, W4>(tx, p, grid, stream);
    default: return launch_nt<64, false, W4>(tx, p, grid, stream);
  }
}

// Resident clusters of `csize` CTAs for the variant a shape launches.
template <bool W4>
static int resident_for(const Shape& s, bool xh, int csize) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (xh) {
    switch (s.NT) {
      case 64: return resident_clusters<64, true, W4>(dev, csize);
      case 128: return resident_clusters<128, true, W4>(dev, csize);
      case 144: return resident_clusters<144, true, W4>(dev, csize);
      case 192: return resident_clusters<192, true, W4>(dev, csize);
      default: return resident_clusters<256, true, W4>(dev, csize);
    }
  }
  switch (s.NT) {
    case 16: return resident_clusters<16, false, W4>(dev, csize);
    case 32: return resident_clusters<32, false, W4>(dev, csize);
    default: return resident_clusters<64, false, W4>(dev, csize);
  }
}

// Whether the wide variant for this tile width can run on the current device.
template <bool W4>
static bool wide_usable(int nt) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaError_t e = nt == 128   ? check_split<128, true, W4>(dev)
                  : nt == 144 ? check_split<144, true, W4>(dev)
                  : nt == 192 ? check_split<192, true, W4>(dev)
                              : check_split<256, true, W4>(dev);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess;
}

// Work split.  Four ways to deal the (tile, K block) items over one CTA per
// SM, chosen by a cost in K blocks: the most blocks any CTA streams plus a
// penalty for each cross-CTA reduction a CTA takes part in.  Measured (a
// globaltimer trace per phase): a block takes ~0.4 us at tiles of <= 64
// tokens and ~0.8 us at 128 or more (the MMA rate), the integer atomics,
// fence, counter and read-back that end a split tile 2-6 us, i.e. ~5 blocks'
// time, and a cluster's exchange through distributed shared memory well
// under a microsecond.
//  * a cluster of C CTAs per tile (grid = tiles x C, all clusters resident at
//    once), each CTA one K part, the parts summed in shared memory;
//  * P parts per tile (grid = tiles x P, tiles <= SMs): every CTA owns one
//    segment of one tile (P = 1: whole tiles, no reduction at all);
//  * whole tiles in contiguous runs (tiles > SMs: each CTA takes
//    ceil(tiles / SMs) or one fewer, no reduction);
//  * equal contiguous ranges of items (stream-K): balanced, but most CTAs
//    publish a partial tile twice, once in the middle of their range.
struct Split {
  int grid;
  int tile_ranges;
  int csize;
};

template <bool W4>
static Split split_of(const Shape& s, bool xh, int sms) {
  // a split tile's atomics and read-back cost ~5 blocks' time at narrow
  // tiles, ~10 at tiles of 192 or more tokens (measured 5-12 us at 256)
  const long long rho = s.NT >= 192 ? 10 : 5, rho_cluster = 1;
  const long long total = (long long)s.tiles * s.KB;
  Split best{(int)std::min<long long>(total, sms), 0, 1};
  long long best_cost = (total + sms - 1) / sms + (s.tiles < total ? 2 * rho : 0);
  if (s.tiles <= sms) {
    const int pmax = std::min(sms / s.tiles, s.KB);
    for (int P = 1; P <= pmax; ++P) {
      const long long cost = (s.KB + P - 1) / P + (P > 1 ? rho : 0);
      if (cost < best_cost) {
        best_cost = cost;
        best = Split{s.tiles * P, 0, 1};
      }
    }
    for (int C = 2; C <= std::min(pmax, 4); ++C) {
      const long long cost = (s.KB + C - 1) / C + rho_cluster;
      if (cost < best_cost && resident_for<W4>(s, xh, C) >= s.tiles) {
        best_cost = cost;
        best = Split{s.tiles * C, 0, C};
      }
    }
  } else {
    const long long cost = (long long)((s.tiles + sms - 1) / sms) * s.KB;
    if (cost <= best_cost) best = Split{sms, 1, 1};
  }
  return best;
}

// `xh_ext` (optional, the one-call entry): the token codes already widened to
// fp16 [M][K] by the quantizer; 64- to 128-token tiles then take them from there.
// `w4`: Wp holds 4-bit packed weights (quasar_pack_weights_w4).
quasar_status_t run(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M, int N, int K,
                    void* Y, int ldy, int32_t* acc_out, void* ws, size_t ws_bytes, cudaStream_t stream,
                    const void* xh_ext = nullptr, bool w4 = false, const skinny::FusedIn* fin = nullptr) {
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
  int32_t* ws_acc = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) + cnt_bytes(M, N, K));
  const size_t xh_off = cnt_bytes(M, N, K) + align256(std::max((size_t)M * N * 4, skinny::slots_bytes(M, N, K)));
  // A few tokens: the register-path kernel (same packed weights, same
  // workspace layout, fewer counters per tile).
  if (skinny::handles(M, N))
    return skinny::run(Xq, sa, Wp, sw, M, N, K, Y, ldy, acc_out, ws_cnt, ws_acc, stream, w4, fin);
  // Wide tiles whose register split the device cannot honour fall back to
  // 64-row tiles (fewer counters and no fp16 copy: the workspace suffices).
  if (s.NT >= 128 && !(w4 ? wide_usable<true>(s.NT) : wide_usable<false>(s.NT))) s = shape_with(M, N, K, 64);

  const bool ext = xh_ext != nullptr && s.NT >= 64;
  const bool xh_path = ext || use_xh(M, N, s);
  uint4* xh = ext ? reinterpret_cast<uint4*>(const_cast<void*>(xh_ext))
              : xh_path ? reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws) + xh_off)
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
  const Split sp = w4 ? split_of<true>(s, xh_path, sms) : split_of<false>(s, xh_path, sms);
  const int grid = sp.grid;
  p.tile_ranges = sp.tile_ranges;
  p.csize = sp.csize;
  // Weight stages issued before the dependency wait.  Measured (graph
  // replays, cold L2): at tiles of <= 64 tokens one stage is 0-6% faster
  // than a full ring (less traffic queued ahead of the token loads); wider
  // tiles stream 1-3% faster with the full ring.
  p.pre = s.NT <= 64 ? 1 : 1 << 30;
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
      e = w4 ? launch_tc<true>(s.NT, true, tx, p, grid, stream) : launch_tc<false>(s.NT, true, tx, p, grid, stream);
    // leave the workspace zero-filled (the internal fp16 copy is scratch of this call)
    if (e == cudaSuccess && !ext) e = cudaMemsetAsync(xh, 0, (size_t)M * K * 2, stream);
    return cuda_status(e);
  }
  e = w4 ? launch_tc<true>(s.NT, false, tx, p, grid, stream) : launch_tc<false>(s.NT, false, tx, p, grid, stream);
  return cuda_status(e);
}

// ------------------------------------------------------ fused activation path
//
// Smooth + quantize (A2) and the linear (A3 + A4) in one call, the codes and
// scales kept in the workspace's scratch tail.  On the register path (up to
// 24 tokens, 32 on layers of <= 8192 rows: skinny::handles) the launch
// quantizes the rows itself (one launch); otherwise the quantizer writes them
// and the linear reads them (two launches, the second overlapping the first
// through programmatic dependent launch).

// The linear's workspace, then the quantizer's codes and scales, then (64- to
// 128-token tiles) the codes again as fp16 for the linear's token operand.
static bool fused_xh(int M, int N, int K) { return !skinny::handles(M, N) && shape_of(M, N, K).NT >= 64; }

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
  if (skinny::handles(M, N)) {
    const skinny::FusedIn fin{X, ldx, smooth};
    return run(xq, sa, Wp, sw, M, N, K, Y, ldy, nullptr, ws, lin, stream, nullptr, false, &fin);
  }
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

size_t quasar_w8a8_linear_workspace_zeroed_bytes(int M, int N, int K) {
  return quasar::gemm::zeroed_bytes(M, N, K);
}

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
  // 4-bit weight blocks on both kernels: the register path for a few tokens
  // (skinny::handles), the tcgen05 kernel (nibbles widened by the converters)
  // above.
  return quasar::gemm::run(Xq, sa, Wp4, sw, M, N, K, Y_bf16, ldy, nullptr, workspace, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream), nullptr, true);
}

quasar_status_t quasar_int8_gemm_s32(const int8_t* Xq, const int8_t* Wp, int M, int N, int K, int32_t* acc,
                                     void* workspace, size_t ws_bytes, quasar_stream_t stream) {
  if (!acc && M > 0) return QUASAR_ERR_INVALID_ARG;
  return quasar::gemm::run(Xq, nullptr, Wp, nullptr, M, N, K, nullptr, 0, acc, workspace, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
