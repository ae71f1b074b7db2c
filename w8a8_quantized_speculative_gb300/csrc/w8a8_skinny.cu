// A3 + A4 for a few tokens (M <= 32, see handles()): the W8A8 verify linear
// on the register tensor path.
//
//   acc[m][n] = sum_k Xq[m][k] * Wq[n][k]        exact integer
//   Y[m][n]   = bf16_rne((float(acc) * sa[m]) * sw[n])
//
// Quasar summary pt §2 "Metodologia" steps 3-4 (INT8 matmul, dequantized to
// BF16); pt §1 / zh §1: the verification pass is bound by the weight stream.
//
// Why a second kernel: with a handful of tokens every weight byte meets at
// most 32 token columns, so the tensor work per byte is tiny and what counts
// is how fast the SM can turn staged INT8 weights into MMA operands.  A
// tcgen05.mma of M = 128, K = 16 costs ~114 cycles for any N <= 192
// (measured with quasar_probe_tensor_rate), i.e. ~18 weight bytes per cycle
// before the weights are even widened into TMEM.  The warp-level m16n8k16
// fp16 MMA covers ~1014 MAC/clk/SM on sm_103a (same probe) and takes its
// weight operand straight from registers: at M <= 8 that is ~127 weight
// bytes per cycle, at M = 32 still ~32, against the ~22 bytes per cycle an
// SM must stream for HBM rate.
// So for a few tokens the weights go HBM -> shared memory (1-D bulk copies of
// the same packed blocks the tcgen05 kernel reads) -> registers (ldmatrix) ->
// fp16 (exact) -> mma.sync, with fp32 accumulators that stay exact integers
// (see RUN_BLOCKS).  Measured, this path is the faster one up to 24 tokens,
// and up to 32 on layers of <= 8192 rows (handles() below is the one place
// that sets the split); the tcgen05 kernel takes larger M.
//
// Work units.  A unit is 64 weight rows (half of a packed 128-row tile: its
// blocks are contiguous 8 KB halves of the 16 KB packed blocks) over all of
// K.  Two CTAs share each SM (~113 KB of shared memory each).  Inside a
// CTA, consumer warp kq owns K bytes [32 kq, 32 kq + 32) of all 64 rows: 4
// row tiles x 2 K steps x NT/8 token tiles of MMAs per block, so each
// token operand is widened once per CTA.  The four K owners of a row tile
// are summed through shared memory once per accumulation run.
//
// Schedules.  A split unit's sums must cross CTAs, and doing that at the end
// of a launch puts a chain of dependent memory round trips after the last
// weight byte, so the exchange is kept off the launch's tail:
//  * few units: a thread-block cluster of C CTAs takes one unit, each CTA a
//    1/C slice of its K blocks; the slices are summed through distributed
//    shared memory between two cluster barriers.
//  * otherwise: the units that do not divide evenly over the CTAs are split
//    stream-K over all CTAs and done first; each CTA then streams whole
//    units.  A split unit is summed without atomics on the data: each
//    contributor stores its integer partial sums into a slot of its own in
//    the workspace and counts its K blocks on a per-(unit, warp) counter; the
//    warp that completes the count adds up the slots of every contributor and
//    runs the epilogue, while the whole units still stream.
//
// K order inside an MMA.  ldmatrix hands thread (g, c) of a warp the four
// consecutive bytes 4c..4c+3 of row g of an 8 x 16-byte matrix.  The MMA's
// K slots 2c, 2c+1 take bytes 4c, 4c+1 and slots 2c+8, 2c+9 take bytes
// 4c+2, 4c+3, for the weights and for the tokens alike.  A dot product does
// not depend on the order of its terms, so this permutation of K leaves
// every sum unchanged.
#include <algorithm>

#include "quasar_common.cuh"

namespace quasar {
namespace skinny {

constexpr int TILE_ROWS = 128;    // rows of a packed weight tile
constexpr int UM = 64;            // rows of a work unit (half a tile)
constexpr int BK = 128;           // K bytes per block
constexpr int PACKED_BLOCK = TILE_ROWS * BK;   // 16 KB packed block
constexpr int HALF_BYTES = UM * BK;            // 8 KB: one unit's part of a block
// 4-bit weights (W4): 64 bytes per row, the same 128 x 128 blocks at half
// the size (8 KB, a unit's half 4 KB).
template <bool W4>
__host__ __device__ constexpr int packed_block() { return W4 ? PACKED_BLOCK / 2 : PACKED_BLOCK; }
template <bool W4>
__host__ __device__ constexpr int half_bytes() { return W4 ? HALF_BYTES / 2 : HALF_BYTES; }
constexpr int KQ = 4;             // K quarters (32 K = 2 MMA K steps each)
constexpr int UT = UM / 16;       // row tiles per unit
constexpr int CWARPS = KQ;        // consumer warps: warp w owns K quarter w of all rows, finalizes row tile w
constexpr int PRODUCER_WARP = CWARPS;
constexpr int THREADS = 32 * (CWARPS + 1);
constexpr int RED_BAR = 1;        // named barrier of the consumer warps
constexpr int MAX_CTAS = 320;     // grid cap (two CTAs per SM); sizes the partial-sum slots
constexpr int MAX_CSIZE = 8;      // CTAs per cluster (K slices of one unit), portable cluster limit
constexpr int CNT_PER_UNIT = 8;   // workspace counters per unit (16 per 128-row tile)
constexpr int SMEM_CAP = 113 * 1024;   // two CTAs per SM
constexpr int G = 2;              // K blocks per pipeline stage (one handshake per pair)
// A warp adds 32 products per block into each fp32 accumulator, each product
// at most 127^2 = 16129 in magnitude: 32 blocks x 32 x 16129 < 2^24, so over
// a run of <= 32 blocks every partial sum is an exact integer in fp32.
constexpr int RUN_BLOCKS = 32;
static_assert(RUN_BLOCKS % 2 == 0, "runs end on a stage boundary");

// RIR: the run-end reduction buffer overlays the stage ring.  Only valid
// when a CTA's single accumulation run ends after its last block (the ring
// is then idle): the cluster schedule with K slices of <= RUN_BLOCKS blocks.
// The space it frees becomes more stages in flight.
template <int NT8, bool RIR = false, bool W4 = false>
struct Cfg {
  static constexpr int NT = 8 * NT8;                        // token columns (padded to 8)
  static constexpr int NH = NT8;                            // token tiles of one finalizer share
  static constexpr int XB = NT * BK;                        // INT8 token tile of a block
  static constexpr int HB = half_bytes<W4>();               // a unit's weight bytes of a block
  static constexpr int BLK = HB + XB;                       // one block: weight half + token tile
  static constexpr int STAGE = G * BLK;                     // multiple of 1024 (swizzle atoms)
  static constexpr int RED = UT * KQ * NT8 * 32 * 16;       // fp32 partials: [row tile][kq][token tile][lane]
  static constexpr int FIN = UT * NT8 * 32 * 16;            // int32 run sums: [row tile][token tile][lane]
  static constexpr int SLOT = UT * NT8 * 32;                // int4 per partial-sum slot (64 rows x NT)
  static constexpr int SCL = 1024;                          // staged scales: sa[32], sw of 2 units
  static constexpr int FIXED = 1024 + (RIR ? 0 : RED) + FIN + SCL + 256;
  static constexpr int S_FIT = (SMEM_CAP - FIXED) / STAGE;
  static constexpr int S = S_FIT < 12 ? S_FIT : 12;         // stages in flight
  static constexpr int SMEM = FIXED + S * STAGE;
  static_assert(BLK % 1024 == 0, "block alignment");
  static_assert(S >= 2, "pipeline depth");
  static_assert(SMEM <= SMEM_CAP, "two CTAs per SM");
  static_assert(!RIR || RED <= S * STAGE, "reduction buffer fits in the ring");
};

// The one-call entry's activations: X [M][ldx] BF16 and the smoothing vector.
struct FusedIn {
  const void* X;
  int ldx;
  const float* smooth;
};

struct Params {
  const uint8_t* wp;  // packed weights, [n_tiles][KB][128 rows][128 B]
  const float* sa;
  const float* sw;
  int M, N, K;
  int KB;           // K blocks per unit
  int mode;         // 0: split units stream-K, then whole units; 1: cluster per unit
  int csize;        // mode 1: CTAs per cluster (K slices per unit)
  int split_units;  // mode 0: units [0, split_units) are split stream-K ...
  int total1;       //   ... over their split_units * KB blocks
  int whole_per;    // mode 0: whole units per CTA, after the split units
  int pre;          // weight stages issued before waiting for the previous kernel
  __nv_bfloat16* Y;
  int ldy;
  int32_t* acc_out;   // int32 mode when non-null
  int4* slots;        // [grid][2] partial sums, each [row tile][token tile][lane] int4
  uint32_t* ws_cnt;   // [units][8] K-block counters per finalizer warp, zero between calls
  unsigned int* err;
  unsigned long long limit_ns;
  // One-call entry (X non-null): the launch smooths and quantizes the token
  // rows itself (row r by CTA r, r + grid, ...) into xq / sa (the buffers the
  // tensor map and `sa` point at), publishes them on a workspace counter and
  // loads no token tile before all M rows are published.
  const uint16_t* X;  // BF16 activations [M][ldx]
  const float* smooth;
  int ldx;
  int8_t* xq;         // codes out, [M][K]
  float* sa_out;      // scales out (== sa)
  uint32_t* qflag;    // [0] rows published, [1] waiters past the wait; zero between calls
};

// First block of CTA c, and the CTA whose range holds block b, for the even
// split of `total` items over `grid` CTAs.  The host guarantees
// (total + 1) * (grid + 1) < 2^32, so 32-bit unsigned arithmetic is exact
// (64-bit division is emulated and far slower).
QUASAR_DEVICE_INLINE int range_begin(int c, int total, int grid) {
  return (int)(((unsigned)c * (unsigned)total) / (unsigned)grid);
}
QUASAR_DEVICE_INLINE int cta_of_block(int b, int total, int grid) {
  return (int)(((unsigned)(b + 1) * (unsigned)grid + (unsigned)total - 1u) / (unsigned)total) - 1;
}

// One CTA's work: split items [s0, s1) (item i = K block i % KB of unit
// i / KB), then whole units [w0, w1).
struct Sched {
  int s0, s1, w0, w1;
};

QUASAR_DEVICE_INLINE Sched schedule_of(int c, int grid, const Params& p) {
  Sched sc;
  if (p.mode == 1) {
    const int u = c / p.csize, q = c % p.csize;
    sc.s0 = u * p.KB + (q * p.KB) / p.csize;
    sc.s1 = u * p.KB + ((q + 1) * p.KB) / p.csize;
    sc.w0 = sc.w1 = 0;
  } else {
    sc.s0 = range_begin(c, p.total1, grid);
    sc.s1 = range_begin(c + 1, p.total1, grid);
    sc.w0 = p.split_units + c * p.whole_per;
    sc.w1 = sc.w0 + p.whole_per;
  }
  return sc;
}

// Walks a schedule one stage (g <= G consecutive K blocks) per step.
// Segments (the CTA's blocks of one unit within a phase) and accumulation
// runs (<= RUN_BLOCKS blocks of a segment, RUN_BLOCKS a multiple of G) are
// contiguous and always end on a stage boundary.
struct Walk {
  int u, kb, kb_first, left, left2, w_next, phase, g;
  __device__ Walk(const Sched& sc, int KB) {
    if (sc.s1 > sc.s0) {
      phase = 1;
      u = sc.s0 / KB;
      kb = kb_first = sc.s0 % KB;
      left = sc.s1 - sc.s0;
      left2 = (sc.w1 - sc.w0) * KB;
    } else {
      phase = 2;
      u = sc.w0;
      kb = kb_first = 0;
      left = (sc.w1 - sc.w0) * KB;
      left2 = 0;
    }
    w_next = sc.w0;
    size(KB);
  }
  __device__ void size(int KB) {
    g = G;
    if (g > left) g = left;
    if (g > KB - kb) g = KB - kb;
  }
  __device__ bool more() const { return left > 0; }
  __device__ bool seg_last(int KB) const { return left == g || kb + g == KB; }
  __device__ bool run_last(int KB) const { return seg_last(KB) || ((kb - kb_first + g) % RUN_BLOCKS) == 0; }
  __device__ void next(int KB) {
    left -= g;
    kb += g;
    if (kb == KB) {
      kb = 0;
      kb_first = 0;
      ++u;
    }
    if (left == 0 && left2 > 0) {   // enter the whole units
      phase = 2;
      u = w_next;
      kb = kb_first = 0;
      left = left2;
      left2 = 0;
    }
    if (left > 0) size(KB);
  }
};

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

// Global address of unit u's half of packed block (tile u / 2, K block kb).
template <bool W4>
QUASAR_DEVICE_INLINE const uint8_t* unit_block(const Params& p, int u, int kb) {
  return p.wp + ((size_t)(u >> 1) * p.KB + kb) * packed_block<W4>() + (size_t)(u & 1) * half_bytes<W4>();
}

QUASAR_DEVICE_INLINE void ldsm_x4(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2, uint32_t& d3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
               : "r"(addr)
               : "memory");
}

QUASAR_DEVICE_INLINE uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// int4 at the same shared-memory offset in cluster CTA `rank`.
QUASAR_DEVICE_INLINE int4 ld_dsmem_int4(const void* local, uint32_t rank) {
  const uint32_t remote = map_to_rank(local, rank);
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// D += A (16 x 16, fp16, row) * B (16 x 8, fp16, col), fp32 accumulate.
QUASAR_DEVICE_INLINE void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------ A2 inside the launch
//
// Eight BF16 values (one 16-byte load) -> fp32, exactly.
QUASAR_DEVICE_INLINE void bf16x8_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Smooth + quantize of token row r by the 128 consumer threads, with the
// stand-alone quantizer's arithmetic step for step (so the codes and the
// scale are bit-identical to it): xs = fp32(x) * smooth[k] rounded once,
// amax = max |xs| over the row, inv = 127 / amax, code = clamp(rne(xs * inv),
// -127, 127), sa = amax / 127 (codes and scale 0 for an all-zero row).
// pt §2 step 2 (per-token symmetric INT8 of the smoothed activations).
QUASAR_DEVICE_INLINE void quantize_row(const Params& p, int r, float* red4) {
  constexpr int T = CWARPS * 32;
  constexpr int U = 4;   // 8-value vectors per thread and round (a row of <= 4096 values is one round)
  const int t = threadIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(p.X + (size_t)r * p.ldx);
  const float4* sm = reinterpret_cast<const float4*>(p.smooth);
  const int nvec = p.K / 8;
  const bool one_round = nvec <= U * T;   // then the smoothed values stay in registers for the codes
  float x[U][8];
  float amax = 0.f;
  auto load_round = [&](int v0) {
    uint4 raw[U];
    float4 s[2 * U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int v = v0 + i * T + t;
      if (v < nvec) {
        raw[i] = __ldg(src + v);
        s[2 * i] = __ldg(sm + 2 * v);
        s[2 * i + 1] = __ldg(sm + 2 * v + 1);
      }
    }
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (v0 + i * T + t >= nvec) continue;
      float xv[8];
      bf16x8_f32(raw[i], xv);
      const float sv[8] = {s[2 * i].x, s[2 * i].y, s[2 * i].z, s[2 * i].w,
                           s[2 * i + 1].x, s[2 * i + 1].y, s[2 * i + 1].z, s[2 * i + 1].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) x[i][e] = __fmul_rn(xv[e], sv[e]);
    }
  };
  for (int v0 = 0; v0 < nvec; v0 += U * T) {
    load_round(v0);
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (v0 + i * T + t >= nvec) continue;
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[i][e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((t & 31) == 0) red4[t >> 5] = amax;
  named_barrier_or(RED_BAR, T, 0u);
  amax = red4[0];
#pragma unroll
  for (int w = 1; w < CWARPS; ++w) amax = fmaxf(amax, red4[w]);
  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  if (t == 0) p.sa_out[r] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(p.xq + (size_t)r * p.K);
  for (int v0 = 0; v0 < nvec; v0 += U * T) {
    if (!one_round) load_round(v0);   // longer rows: the round again (L1 / L2)
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int v = v0 + i * T + t;
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
      dst[v] = make_uint2(packed[0], packed[1]);
    }
  }
  named_barrier_or(RED_BAR, T, 0u);   // red4 is free again; every store of the row is issued
}

QUASAR_DEVICE_INLINE uint32_t ld_relaxed_u32(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

QUASAR_DEVICE_INLINE void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

QUASAR_DEVICE_INLINE float ld_relaxed_f32(const float* ptr) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(ptr) : "memory");
  return v;
}

QUASAR_DEVICE_INLINE void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bounded wait (the copy thread of each CTA) until every token row is
// published: relaxed polls of the count, then one acquire fence.  Every CTA
// of the launch is resident at once (the host sizes the grid to one wave),
// so the rows' writers always run.  Gives up like mbar_wait.  A thread that
// saw the count then counts itself past the wait; the last of the grid's
// waiters zeroes both counters for the next call.  (One waiter per CTA: the
// consumers learn of the rows through the first stage's barrier, which the
// copy thread fills only after its wait; with a second poller per CTA the
// attention step ran 0.9 us slower.)
QUASAR_DEVICE_INLINE bool wait_rows(const Params& p, volatile int* abort_flag) {
  bool ok = true;
  if (ld_relaxed_u32(p.qflag) < (uint32_t)p.M) {
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      if (ld_relaxed_u32(p.qflag) >= (uint32_t)p.M) break;
      if ((it & 15u) == 0) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (globaltimer_ns() - t0 > p.limit_ns) {
          *abort_flag = 1;
          if (p.err) atomicCAS(p.err, 0u, SITE_SKINNY_ROWS | ((blockIdx.x & 0xFFFFu) << 16));
          ok = false;
          break;
        }
      }
    }
  }
  fence_acq_rel_gpu();
  if (ok && atomicAdd(p.qflag + 1, 1u) == gridDim.x - 1u) {
    p.qflag[0] = 0u;
    p.qflag[1] = 0u;
  }
  return ok;
}

// Publishes this CTA's `rows` finished token rows (one thread, after a
// barrier with the threads that stored them): a release add, cumulative over
// those stores.
QUASAR_DEVICE_INLINE void publish_rows(const Params& p, uint32_t rows) {
  fence_proxy_async_global();   // the tensor copies of other CTAs read the rows
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p.qflag), "r"(rows) : "memory");
}

// A finalizer warp's share of a unit is row tile mt and every token tile:
// lane holds int4 v[ni] (nh = 0 below), whose element j is row 8 (j >> 1) + g
// of the row tile, token 8 ni + 2c + (j & 1).
// `sa_s` holds sa of every token (shared memory), `swu` sw of the unit's 64
// rows (shared memory for the CTA's first and last unit, else global).
template <int NT8>
QUASAR_DEVICE_INLINE void epilogue(const Params& p, const int4 (&v4)[Cfg<NT8>::NH], int u, int mt, int nh, int lane,
                                   const float* sa_s, const float* swu) {
  const int g = lane >> 2, c = lane & 3;
  const int nrow0 = u * UM + mt * 16 + g;
  float swr[2] = {0.f, 0.f};
  if (!p.acc_out) {
    swr[0] = swu[mt * 16 + g];
    swr[1] = swu[mt * 16 + g + 8];
  }
#pragma unroll
  for (int h = 0; h < Cfg<NT8>::NH; ++h) {
    const int ni = nh + h;
    if (ni >= NT8) break;
    const int32_t v[4] = {v4[h].x, v4[h].y, v4[h].z, v4[h].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = ni * 8 + 2 * c + (j & 1), n = nrow0 + 8 * (j >> 1);
      if (m >= p.M || n >= p.N) continue;
      if (p.acc_out) {
        p.acc_out[(size_t)m * p.N + n] = v[j];
      } else {
        const float y = __fmul_rn(__fmul_rn(__int2float_rn(v[j]), sa_s[m]), swr[j >> 1]);
        p.Y[(size_t)m * p.ldy + n] = __float2bfloat16_rn(y);
      }
    }
  }
}

// Slot of contributor cc for split unit u: a contributor's segment of a split
// unit is the first segment of its split range (slot 0) or the last (slot 1);
// every one is partial.  Points at lane's int4 of the share's token tile nh.
template <int NT8>
QUASAR_DEVICE_INLINE int4* slot_ptr(const Params& p, int cc, int u, int mt, int nh, int lane, int grid) {
  const int first_u = range_begin(cc, p.total1, grid) / p.KB;
  return p.slots + ((size_t)cc * 2 + (first_u == u ? 0 : 1)) * Cfg<NT8>::SLOT + ((size_t)mt * NT8 + nh) * 32 + lane;
}

// Sum of every contributor's slot for this warp's share of split unit u
// (loads only: four contributors in flight at a time).
template <int NT8>
QUASAR_DEVICE_INLINE void load_slots(const Params& p, int u, int mt, int nh, int lane, int grid,
                                     int4 (&s)[Cfg<NT8>::NH]) {
  constexpr int NH = Cfg<NT8>::NH;
  const int c_lo = cta_of_block(u * p.KB, p.total1, grid);
  const int c_hi = cta_of_block((u + 1) * p.KB - 1, p.total1, grid);
#pragma unroll
  for (int h = 0; h < NH; ++h) s[h] = make_int4(0, 0, 0, 0);
  for (int c0 = c_lo; c0 <= c_hi; c0 += 4) {
    int4 v[4][NH];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int4* slot = slot_ptr<NT8>(p, c0 + q <= c_hi ? c0 + q : c_hi, u, mt, nh, lane, grid);
#pragma unroll
      for (int h = 0; h < NH; ++h)
        v[q][h] = (c0 + q <= c_hi && nh + h < NT8) ? __ldcg(slot + h * 32) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        s[h].x += v[q][h].x;
        s[h].y += v[q][h].y;
        s[h].z += v[q][h].z;
        s[h].w += v[q][h].w;
      }
  }
}

// Each slot share is read exactly once (by the warp that completes the unit)
// and zeroed after the read, so the workspace is left as it was found.
template <int NT8>
QUASAR_DEVICE_INLINE void zero_slots(const Params& p, int u, int mt, int nh, int lane, int grid) {
  const int c_lo = cta_of_block(u * p.KB, p.total1, grid);
  const int c_hi = cta_of_block((u + 1) * p.KB - 1, p.total1, grid);
  for (int cc = c_lo; cc <= c_hi; ++cc) {
    int4* slot = slot_ptr<NT8>(p, cc, u, mt, nh, lane, grid);
#pragma unroll
    for (int h = 0; h < Cfg<NT8>::NH; ++h)
      if (nh + h < NT8) __stcg(slot + h * 32, make_int4(0, 0, 0, 0));
  }
}

// Publish partial segments: one fence for this warp's slot stores, then the
// K-block count of each segment (unit ua with na blocks, and unit ub with nb
// blocks when ub >= 0); a warp whose count completes a unit sums the unit's
// slots and runs its epilogue.  Both units' slots are loaded before either
// epilogue so that their latencies overlap.
template <int NT8>
QUASAR_DEVICE_INLINE void count_segments(const Params& p, int ua, int na, int ub, int nb, int warp, int mt, int nh,
                                         int lane, int grid, const float* sa_s, const float* swa,
                                         const float* swb) {
  constexpr int NH = Cfg<NT8>::NH;
  __threadfence();
  __syncwarp();
  uint32_t last_mask = 0;
  if (lane == 0) {
    const uint32_t old_a = atomicAdd(&p.ws_cnt[(size_t)ua * CNT_PER_UNIT + warp], (uint32_t)na);
    const uint32_t old_b = (ub >= 0) ? atomicAdd(&p.ws_cnt[(size_t)ub * CNT_PER_UNIT + warp], (uint32_t)nb) : 0u;
    if (old_a + (uint32_t)na == (uint32_t)p.KB) last_mask |= 1u;
    if (ub >= 0 && old_b + (uint32_t)nb == (uint32_t)p.KB) last_mask |= 2u;
  }
  last_mask = __shfl_sync(0xffffffffu, last_mask, 0);
  if (!last_mask) return;
  __threadfence();
  int4 va[NH], vb[NH];
  if (last_mask & 1u) load_slots<NT8>(p, ua, mt, nh, lane, grid, va);
  if (last_mask & 2u) load_slots<NT8>(p, ub, mt, nh, lane, grid, vb);
  if (last_mask & 1u) {
    zero_slots<NT8>(p, ua, mt, nh, lane, grid);
    epilogue<NT8>(p, va, ua, mt, nh, lane, sa_s, swa);
    if (lane == 0) p.ws_cnt[(size_t)ua * CNT_PER_UNIT + warp] = 0u;   // ready for the next call
  }
  if (last_mask & 2u) {
    zero_slots<NT8>(p, ub, mt, nh, lane, grid);
    epilogue<NT8>(p, vb, ub, mt, nh, lane, sa_s, swb);
    if (lane == 0) p.ws_cnt[(size_t)ub * CNT_PER_UNIT + warp] = 0u;
  }
}

// One K block of this warp's work: its two K steps of the unit's 64 rows
// against every token tile.  Token operands: row n = 8 ni + g of the
// swizzled tile sits at n * 128, chunk ch at (ch ^ (n & 7)) * 16.

template <int NT8, bool W4>
QUASAR_DEVICE_INLINE void consume_block(uint32_t st, uint32_t a_off, uint32_t b_off, float (&acc)[UT][NT8][4]) {
  if constexpr (W4) {
    // 4-bit weights: one ldmatrix word holds a row's 4 K values of both
    // 16-K steps (low nibbles: the first, high nibbles: the second), each
    // stored as code + 8.
    uint32_t bq[2][NT8][2];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni)
        s8x4_to_f16x4(lds32(st + (b_off ^ (ks << 4)) + (uint32_t)(ni * 8 * BK)), bq[ks][ni][0], bq[ks][ni][1]);
#pragma unroll
    for (int i2 = 0; i2 < UT / 2; ++i2) {
      uint32_t d[4];
      ldsm_x4(st + a_off + (uint32_t)(i2 * 32 * 64), d[0], d[1], d[2], d[3]);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint32_t a0, a1, a2, a3;
          n4x4_to_f16x4(ks ? (d[2 * i] >> 4) & 0x0F0F0F0Fu : d[2 * i] & 0x0F0F0F0Fu, a0, a2);
          n4x4_to_f16x4(ks ? (d[2 * i + 1] >> 4) & 0x0F0F0F0Fu : d[2 * i + 1] & 0x0F0F0F0Fu, a1, a3);
#pragma unroll
          for (int ni = 0; ni < NT8; ++ni)
            mma_16816(acc[2 * i2 + i][ni], a0, a1, a2, a3, bq[ks][ni][0], bq[ks][ni][1]);
        }
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t bq[NT8][2];
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni)
        s8x4_to_f16x4(lds32(st + (b_off ^ (ks << 4)) + (uint32_t)(ni * 8 * BK)), bq[ni][0], bq[ni][1]);
#pragma unroll
      for (int i2 = 0; i2 < UT / 2; ++i2) {
        uint32_t d[4];
        ldsm_x4(st + (a_off ^ (ks << 4)) + (uint32_t)(i2 * 32 * BK), d[0], d[1], d[2], d[3]);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint32_t a0, a1, a2, a3;
          u8x4_to_f16x4(d[2 * i], a0, a2);       // rows g: K slots 2c.. (bytes 4c, 4c+1), 2c+8.. (4c+2, 4c+3)
          u8x4_to_f16x4(d[2 * i + 1], a1, a3);   // rows g + 8
#pragma unroll
          for (int ni = 0; ni < NT8; ++ni)
            mma_16816(acc[2 * i2 + i][ni], a0, a1, a2, a3, bq[ni][0], bq[ni][1]);
        }
      }
    }
  }
}

template <int NT8, bool RIR, bool W4>
__global__ void __launch_bounds__(THREADS, 2)
w8a8_skinny_kernel(const __grid_constant__ CUtensorMap tmX, const Params p) {
  using C = Cfg<NT8, RIR, W4>;
  constexpr int NH = C::NH;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;                                     // S x [W half 8 KB | X NT x 128 B]
  constexpr int RED_OWN = RIR ? 0 : C::RED;                  // bytes of a separate reduction buffer
  float4* red = reinterpret_cast<float4*>(RIR ? stages : smem + C::S * C::STAGE);
  int4* fin = reinterpret_cast<int4*>(smem + C::S * C::STAGE + RED_OWN);
  float* sa_s = reinterpret_cast<float*>(smem + C::S * C::STAGE + RED_OWN + C::FIN);   // [32]
  float* sw_s = sa_s + 32;                                                                // [2][64]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::S * C::STAGE + RED_OWN + C::FIN + C::SCL);
  uint64_t* empty = full + C::S;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::S);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CWARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == PRODUCER_WARP && lane == 0) prefetch_tmap(&tmX);
  __syncthreads();

  const int grid = (int)gridDim.x;
  const int KB = p.KB;
  const Sched sc = schedule_of((int)blockIdx.x, grid, p);

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      // Weights do not depend on the previous kernel: issue the first p.pre
      // stages before waiting for it (the host picks the depth).
      int pre = 0;
      {
        Walk w(sc, KB);
        for (; pre < C::S && pre < p.pre && w.more(); ++pre, w.next(KB)) {
          mbar_arrive_expect_tx(&full[pre], (uint32_t)(w.g * C::BLK));
          for (int b = 0; b < w.g; ++b)
            bulk_load(stages + pre * C::STAGE + b * C::BLK, unit_block<W4>(p, w.u, w.kb + b), C::HB, &full[pre],
                      pol_w);
        }
      }
      pdl_wait();  // token codes (or X) come from the previous kernel
      bool rows_ok = true;
      if (p.X) {
        // This launch quantizes the tokens: no token tile before every row is
        // published.  (Filling the rest of the weight ring here instead was
        // slower: the weight requests delay the rows' own loads.)
        rows_ok = wait_rows(p, abort_flag);
        fence_proxy_async_global();   // the rows were written by generic stores; the tensor copies read them
      }
      Walk w(sc, KB);
      Ring<C::S> rg;
      int issued = 0;
      for (; w.more(); w.next(KB), rg.next(), ++issued) {
        // After a failed wait only the stages already in flight are
        // completed (their token tiles read whatever is there), so that
        // nothing is left in flight.
        if (!rows_ok && issued >= pre) break;
        uint8_t* st = stages + rg.s * C::STAGE;
        if (issued >= pre) {
          if (!mbar_wait(&empty[rg.s], rg.ph ^ 1u, abort_flag, p.err, SITE_SKINNY_EMPTY, p.limit_ns)) break;
          mbar_arrive_expect_tx(&full[rg.s], (uint32_t)(w.g * C::BLK));
          for (int b = 0; b < w.g; ++b)
            bulk_load(st + b * C::BLK, unit_block<W4>(p, w.u, w.kb + b), C::HB, &full[rg.s], pol_w);
        }
        for (int b = 0; b < w.g; ++b)
          tma_load_2d(st + b * C::BLK + C::HB, &tmX, (w.kb + b) * BK, 0, &full[rg.s], pol_x);
      }
      // Never leave with copies in flight.
      for (int s = 0; s < C::S && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / C::S) * C::S;
        volatile int dummy = 0;
        mbar_wait(&full[s], (uint32_t)(last / C::S) & 1u, &dummy, p.err, SITE_SKINNY_DRAIN, p.limit_ns);
      }
    }
    __syncwarp();
    if (p.mode == 1) {   // the consumers' two cluster barriers
      cluster_sync_full();
      cluster_sync_exec();
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int kq = warp;              // K bytes [32 kq, 32 kq + 32) of each block, all 64 rows
  const int g = lane >> 2, c = lane & 3;
  const int mt_f = warp;            // finalizer share: row tile mt_f, every token tile
  const int nh = 0;
  pdl_wait();                       // scales and workspace belong to the previous kernel until here
  bool bad = false;
  if (p.X) {
    // A2 for this CTA's token rows, published with one count per CTA.  The
    // consumers then need nothing until their first full stage, which the
    // copy thread fills only after every row is published.
    float* red4 = reinterpret_cast<float*>(fin);
    int rows = 0;
    for (int r = (int)blockIdx.x; r < p.M; r += grid, ++rows) quantize_row(p, r, red4);
    if (threadIdx.x == 0) {
      if (rows > 0) publish_rows(p, (uint32_t)rows);
    }
    named_barrier_or(RED_BAR, CWARPS * 32, 0u);
  }
  const int u_first = (sc.s1 > sc.s0) ? sc.s0 / KB : sc.w0;
  const int u_last = (sc.w1 > sc.w0) ? sc.w1 - 1 : (sc.s1 - 1) / KB;
  const int u_first1 = sc.s0 / KB;  // first unit of the split range (its slot 0)
  // Stage the dequantization scales the epilogues will need: every token's
  // sa (in the one-call launch after the first full stage, below), and sw of
  // the first and last unit of this CTA (read after the first run-end
  // barrier, which orders these stores).
  if (!p.acc_out) {
    for (int i = threadIdx.x; i < 32 + 2 * UM; i += CWARPS * 32) {
      if (i < 32) {
        if (!p.X) sa_s[i] = (i < p.M) ? __ldg(&p.sa[i]) : 0.f;
      } else {
        const int r = i - 32;
        const int n = (r < UM ? u_first : u_last) * UM + (r & (UM - 1));
        sw_s[r] = (n < p.N) ? __ldg(&p.sw[n]) : 0.f;
      }
    }
  }

  float acc[UT][NT8][4];
#pragma unroll
  for (int i = 0; i < UT; ++i)
#pragma unroll
    for (int n = 0; n < NT8; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][n][j] = 0.f;
  // Finished integer sums of this warp's finalizer share, kept in shared
  // memory (touched once per run): token tile h at share[h * 32].
  int4* share = fin + ((size_t)mt_f * NT8 + nh) * 32 + lane;
#pragma unroll
  for (int h = 0; h < NH; ++h)
    if (nh + h < NT8) share[h * 32] = make_int4(0, 0, 0, 0);

  // Per-lane address parts.  ldmatrix over one K step of 32 rows: lanes
  // 8i..8i+7 give rows 8i..8i+7, i.e. matrix i = (row tile i >> 1, row half
  // i & 1); the next 32 rows are 32 * BK further.  Rows keep their swizzle
  // phase because units start at a multiple of 8 rows.  The second K step's
  // chunk differs from the first in bit 0 only, i.e. its offset is the first
  // one's ^ 16.
  // W4: row r of a block is 64 bytes, 16-byte chunk kq (this warp's K
  // quarter) at (kq ^ ((r >> 1) & 3)) * 16.
  const uint32_t a_off = W4 ? (uint32_t)(lane * 64 + ((kq ^ ((lane >> 1) & 3)) << 4))
                            : (uint32_t)(lane * BK + (((2 * kq) ^ (lane & 7)) << 4));
  const uint32_t b_off = (uint32_t)(C::HB + g * BK + (((2 * kq) ^ g) << 4) + 4 * c);
  const uint32_t stages_u32 = smem_u32(stages);

  // Partial segments of the split range (at most two: its first and last)
  // are counted together when the range ends, so that one fence covers both.
  int seg_ua = -1, seg_na = 0, seg_ub = -1, seg_nb = 0;
  // sw of unit u: staged for the CTA's first and last unit.
  auto sw_of = [&](int u) -> const float* {
    return u == u_first ? sw_s : u == u_last ? sw_s + UM : p.sw + (size_t)u * UM;
  };
  Walk w(sc, KB);
  Ring<C::S> r;
  bool sa_late = p.X != nullptr && !p.acc_out;
  for (; w.more(); w.next(KB), r.next()) {
    if (!bad) {
      const bool ok = mbar_wait(&full[r.s], r.ph, abort_flag, p.err, SITE_SKINNY_FULL, p.limit_ns);
      bad = !__all_sync(0xffffffffu, ok);
      if (sa_late && !bad) {
        // The copy thread saw every row published (acquire) before it armed
        // this stage: the token scales written in this launch are visible.
        for (int i = threadIdx.x; i < 32; i += CWARPS * 32) sa_s[i] = (i < p.M) ? ld_relaxed_f32(&p.sa[i]) : 0.f;
      }
      sa_late = false;
    }
    if (!bad) {
      const uint32_t st0 = stages_u32 + (uint32_t)(r.s * C::STAGE);
      // A full pair takes a straight-line path so that the two blocks'
      // loads and MMAs can interleave; a segment's odd tail takes one block.
      if (w.g == G) {
#pragma unroll
        for (int b = 0; b < G; ++b) consume_block<NT8, W4>(st0 + (uint32_t)(b * C::BLK), a_off, b_off, acc);
      } else {
        consume_block<NT8, W4>(st0, a_off, b_off, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[r.s]);
    }
    if (!w.run_last(KB)) continue;

    // ---- end of an accumulation run: sum the four K owners of each row tile.
    // The first barrier also frees the partial buffer of the previous run
    // and carries the abort decision to every consumer warp.
    if (named_barrier_or(RED_BAR, CWARPS * 32, bad ? 1u : 0u)) break;
#pragma unroll
    for (int i = 0; i < UT; ++i)
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni) {
        red[((i * KQ + kq) * NT8 + ni) * 32 + lane] =
            make_float4(acc[i][ni][0], acc[i][ni][1], acc[i][ni][2], acc[i][ni][3]);
        acc[i][ni][0] = acc[i][ni][1] = acc[i][ni][2] = acc[i][ni][3] = 0.f;
      }
    named_barrier_or(RED_BAR, CWARPS * 32, 0u);
    // The four K owners' partials are exact integers of magnitude at most
    // blocks x 32 x 127^2; when a group of them sums below 2^24 it is added
    // in fp32 (exact) before the one conversion to int32: the conversion
    // unit (16 per SM clock) is the slow part of this step.  Groups of four
    // for runs of <= 8 blocks (4 x 8 x 32 x 16129 < 2^24), pairs for <= 16.
    const int run_len = (w.kb + w.g - w.kb_first - 1) % RUN_BLOCKS + 1;
    const int grp = run_len <= 8 ? 4 : run_len <= 16 ? 2 : 1;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const int ni = nh + h;
      if (ni >= NT8) break;
      int4 f = share[h * 32];
      float4 v[KQ];
#pragma unroll
      for (int q = 0; q < KQ; ++q) v[q] = red[((mt_f * KQ + q) * NT8 + ni) * 32 + lane];
      if (grp == 4) {
        f.x += __float2int_rn(((v[0].x + v[1].x) + v[2].x) + v[3].x);
        f.y += __float2int_rn(((v[0].y + v[1].y) + v[2].y) + v[3].y);
        f.z += __float2int_rn(((v[0].z + v[1].z) + v[2].z) + v[3].z);
        f.w += __float2int_rn(((v[0].w + v[1].w) + v[2].w) + v[3].w);
      } else if (grp == 2) {
        f.x += __float2int_rn(v[0].x + v[1].x) + __float2int_rn(v[2].x + v[3].x);
        f.y += __float2int_rn(v[0].y + v[1].y) + __float2int_rn(v[2].y + v[3].y);
        f.z += __float2int_rn(v[0].z + v[1].z) + __float2int_rn(v[2].z + v[3].z);
        f.w += __float2int_rn(v[0].w + v[1].w) + __float2int_rn(v[2].w + v[3].w);
      } else {
#pragma unroll
        for (int q = 0; q < KQ; ++q) {
          f.x += __float2int_rn(v[q].x);
          f.y += __float2int_rn(v[q].y);
          f.z += __float2int_rn(v[q].z);
          f.w += __float2int_rn(v[q].w);
        }
      }
      share[h * 32] = f;
    }
    if (!w.seg_last(KB)) continue;

    // ---- end of this CTA's segment of unit u.
    const int u = w.u;
    const int nb = w.kb + w.g - w.kb_first;
    if (p.mode == 1) break;   // the only segment: summed across the cluster below
    if (nb == KB) {
      int4 v[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) v[h] = (nh + h < NT8) ? share[h * 32] : make_int4(0, 0, 0, 0);
      epilogue<NT8>(p, v, u, mt_f, nh, lane, sa_s, sw_of(u));   // the whole unit
    } else {
      // Partial segment of the split range: store the share into this CTA's
      // slot for it (0 = the range's first segment, 1 = its last).
      int4* slot = p.slots + ((size_t)blockIdx.x * 2 + (u == u_first1 ? 0 : 1)) * C::SLOT +
                   ((size_t)mt_f * NT8 + nh) * 32 + lane;
#pragma unroll
      for (int h = 0; h < NH; ++h)
        if (nh + h < NT8) slot[h * 32] = share[h * 32];
      if (seg_ua < 0) {
        seg_ua = u;
        seg_na = nb;
      } else {
        seg_ub = u;
        seg_nb = nb;
      }
    }
    if (w.phase == 1 && w.left == w.g && seg_ua >= 0) {
      // The split range ends here: publish its partial segments now, while
      // the whole units (if any) still stream.
      count_segments<NT8>(p, seg_ua, seg_na, seg_ub, seg_nb, warp, mt_f, nh, lane, grid, sa_s, sw_of(seg_ua),
                          seg_ub >= 0 ? sw_of(seg_ub) : sw_s);
      seg_ua = -1;
    }
#pragma unroll
    for (int h = 0; h < NH; ++h)
      if (nh + h < NT8) share[h * 32] = make_int4(0, 0, 0, 0);
  }

  if (p.mode == 1) {
    // Cluster split: every CTA of the cluster holds the sums of one K slice of
    // unit u in `fin`.  After the barrier each finalizer share (row tile,
    // token-tile parity) is finished by one CTA (the share of warp w by the
    // CTA of rank w % C), reading the other slices through distributed shared
    // memory; the second barrier keeps every CTA's shared memory alive until
    // those reads are done.
    __syncwarp();
    cluster_sync_full();
    const int csz = p.csize;
    const int rank = (int)blockIdx.x % csz;
    if (!bad && (warp % csz) == rank) {
      int4 v[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) v[h] = (nh + h < NT8) ? share[h * 32] : make_int4(0, 0, 0, 0);
      // Every remote load is issued before any of them is used: one
      // distributed-shared-memory round trip instead of one per load.
      int4 x[MAX_CSIZE - 1][NH];
#pragma unroll
      for (int j = 0; j < MAX_CSIZE - 1; ++j) {
        if (j >= csz - 1) break;
        const int q = rank + 1 + j < csz ? rank + 1 + j : rank + 1 + j - csz;
#pragma unroll
        for (int h = 0; h < NH; ++h)
          if (nh + h < NT8) x[j][h] = ld_dsmem_int4(share + h * 32, (uint32_t)q);
      }
#pragma unroll
      for (int j = 0; j < MAX_CSIZE - 1; ++j) {
        if (j >= csz - 1) break;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          if (nh + h >= NT8) break;
          v[h].x += x[j][h].x;
          v[h].y += x[j][h].y;
          v[h].z += x[j][h].z;
          v[h].w += x[j][h].w;
        }
      }
      epilogue<NT8>(p, v, u_first, mt_f, nh, lane, sa_s, sw_s);
    }
    __syncwarp();
    cluster_sync_exec();
  }
}

// ------------------------------------------------------------------ host side

template <int NT8, bool RIR, bool W4>
static cudaError_t configure(int dev) {
  static int configured[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(w8a8_skinny_kernel<NT8, RIR, W4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<NT8, RIR, W4>::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return cudaSuccess;
}

template <int NT8, bool RIR, bool W4>
static cudaLaunchConfig_t config_of(int grid, int csize, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg<NT8, RIR, W4>::SMEM;
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

// Clusters of `csize` CTAs of the cluster-schedule kernel that the device
// keeps resident at once (0 if unknown); cached per device and cluster size.
template <int NT8, bool W4>
static int resident_clusters(int dev, int csize) {
  static int cache[64][9];
  static bool init[64][9] = {};
  if (dev < 0 || dev >= 64 || csize < 2 || csize > 8) return 0;
  if (!init[dev][csize]) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = config_of<NT8, true, W4>(csize * 16, csize, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, w8a8_skinny_kernel<NT8, true, W4>, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();
    }
    cache[dev][csize] = n;
    init[dev][csize] = true;
  }
  return cache[dev][csize];
}

// CTAs of the stream-K kernel resident per SM (0 if unknown); cached per device.
template <int NT8, bool W4>
static int resident_per_sm(int dev) {
  static int cache[64];
  static bool init[64] = {};
  if (dev < 0 || dev >= 64) return 0;
  if (!init[dev]) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, w8a8_skinny_kernel<NT8, false, W4>, THREADS,
                                                      Cfg<NT8, false, W4>::SMEM) != cudaSuccess) {
      n = 0;
      cudaGetLastError();
    }
    cache[dev] = n;
    init[dev] = true;
  }
  return cache[dev];
}

// Launches the kernel; with p.X set (the launch quantizes its own tokens,
// which needs every CTA resident at once) returns cudaErrorNotSupported
// without launching when the grid would not fit in one wave.
template <int NT8, bool W4>
static cudaError_t launch(const CUtensorMap& tx, Params p, int sms, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = configure<NT8, true, W4>(dev);
  if (e == cudaSuccess) e = configure<NT8, false, W4>(dev);
  if (e != cudaSuccess) return e;
  const int n_units = (p.N + UM - 1) / UM;
  const int slots = std::min(2 * sms, MAX_CTAS);   // two CTAs per SM
  // Few units: one cluster per unit, with the most K slices that keep every
  // cluster resident in one wave; each slice must be one accumulation run.
  int csize = std::min(std::min(MAX_CSIZE, slots / n_units), p.KB);
  while (csize >= 2 && resident_clusters<NT8, W4>(dev, csize) < n_units) --csize;
  if (csize >= 2 && (p.KB + csize - 1) / csize > RUN_BLOCKS) csize = 1;
  cudaLaunchAttribute attr[2];
  // Weight stages a CTA issues before its dependency wait.  Measured (graph
  // replays, cold L2, Qwen3-8B shapes): a full ring floods the memory system
  // just when the previous kernel's last stores and this kernel's first
  // token loads must get through, which costs CTAs with a short K range
  // (qkv, o_proj: 8-11 blocks) 6-11% at 8-24 tokens; CTAs with a long
  // range at a few tokens (down_proj, gate_up: 24-40 blocks, M <= 8) stream
  // 2% faster with the full ring.  So: one stage unless a CTA's range is
  // long and its consumers are fast.
  auto pre_for = [&](int blocks_per_cta) { return (blocks_per_cta <= 16 || p.M > 8) ? 1 : 1 << 30; };
  if (csize >= 2) {
    // (every cluster resident at once: the choice of csize above)
    p.mode = 1;
    p.csize = csize;
    p.split_units = 0;
    p.total1 = 0;
    p.whole_per = 0;
    p.pre = pre_for((p.KB + csize - 1) / csize);
    cudaLaunchConfig_t cfg = config_of<NT8, true, W4>(n_units * csize, csize, stream, attr);
    return cudaLaunchKernelEx(&cfg, w8a8_skinny_kernel<NT8, true, W4>, tx, p);
  }
  p.mode = 0;
  p.csize = 1;
  int grid = slots;
  p.whole_per = n_units / grid;
  p.split_units = n_units - p.whole_per * grid;
  p.total1 = p.split_units * p.KB;
  if (p.whole_per == 0) grid = std::min(grid, p.total1);
  p.pre = pre_for((p.total1 + grid - 1) / std::max(grid, 1) + p.whole_per * p.KB);
  if ((unsigned long long)(p.total1 + 1) * (unsigned long long)(grid + 1) >= (1ull << 32)) return cudaErrorInvalidValue;
  if (p.X && grid > resident_per_sm<NT8, W4>(dev) * sms) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = config_of<NT8, false, W4>(grid, 1, stream, attr);
  return cudaLaunchKernelEx(&cfg, w8a8_skinny_kernel<NT8, false, W4>, tx, p);
}

// Measured (graph replays, cold L2, Qwen3-8B shapes): this path is faster
// than the tcgen05 kernel up to 24 tokens on every layer, and at 25-32
// tokens on layers of up to 8192 rows (qkv 10.4-10.8 against 12.0-12.3 us,
// o_proj 8.3 against 9.7, down_proj 16.8 against 18.3), where one cluster
// per unit applies; wider layers (gate_up, 384 units) stream-K at four token
// tiles slower (34.5 against 30.6 us).
bool handles(int M, int N) { return M >= 1 && (M <= 24 || (M <= 32 && N <= 8192)); }

// Partial-sum slots this kernel may need after the counters: two per CTA,
// each 64 rows x NT int32.  Like the counters they are zero between calls
// (each is zeroed by its reader).
size_t slots_bytes(int M, int N, int K) {
  if (!handles(M, N) || N <= 0 || K <= 0) return 0;
  const long long items = (long long)((N + UM - 1) / UM) * ((K + BK - 1) / BK);
  const long long ctas = std::min<long long>(items, MAX_CTAS);
  return (size_t)ctas * 2 * (size_t)UM * 8 * ((M + 7) / 8) * 4;
}

// Arguments were validated by the caller; ws_cnt holds >= 8 zeroed counters
// per 64-row unit, `slots` slots_bytes() bytes (no initial value needed).
// With `fin` (the one-call entry) the launch first smooths and quantizes
// fin->X into Xq / sa itself; its two row counters are ws_cnt[4] and
// ws_cnt[5], which the stream-K schedule never uses (its counters are
// [unit][finalizer warp < 4]).  If the grid cannot be resident in one wave
// it runs the stand-alone quantizer first instead.
quasar_status_t run(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M, int N, int K,
                    void* Y, int ldy, int32_t* acc_out, uint32_t* ws_cnt, void* slots, cudaStream_t stream,
                    bool w4, const FusedIn* fin) {
  const int nt8 = (M + 7) / 8;
  CUtensorMap tx;
  if (!encode_2d_u8(&tx, Xq, K, M, BK, 8 * nt8)) return QUASAR_ERR_CUDA;
  Params p;
  p.wp = reinterpret_cast<const uint8_t*>(Wp);
  p.sa = sa;
  p.sw = sw;
  p.M = M;
  p.N = N;
  p.K = K;
  p.KB = (K + BK - 1) / BK;
  p.Y = reinterpret_cast<__nv_bfloat16*>(Y);
  p.ldy = ldy;
  p.acc_out = acc_out;
  p.slots = reinterpret_cast<int4*>(slots);
  p.ws_cnt = ws_cnt;
  p.err = device_error_word();
  p.limit_ns = wait_limit_ns();
  p.X = fin ? reinterpret_cast<const uint16_t*>(fin->X) : nullptr;
  p.smooth = fin ? fin->smooth : nullptr;
  p.ldx = fin ? fin->ldx : 0;
  p.xq = const_cast<int8_t*>(Xq);
  p.sa_out = const_cast<float*>(sa);
  p.qflag = ws_cnt + 4;
  if (!p.err) return QUASAR_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return QUASAR_ERR_CUDA;
  auto go = [&]() -> cudaError_t {
    if (w4) {
      switch (nt8) {
        case 1: return launch<1, true>(tx, p, sms, stream);
        case 2: return launch<2, true>(tx, p, sms, stream);
        case 3: return launch<3, true>(tx, p, sms, stream);
        default: return launch<4, true>(tx, p, sms, stream);   // handles() keeps M <= 32
      }
    }
    switch (nt8) {
      case 1: return launch<1, false>(tx, p, sms, stream);
      case 2: return launch<2, false>(tx, p, sms, stream);
      case 3: return launch<3, false>(tx, p, sms, stream);
      default: return launch<4, false>(tx, p, sms, stream);
    }
  };
  cudaError_t e = go();
  if (e == cudaErrorNotSupported && p.X) {
    const quasar_status_t sq = quasar_smooth_quant_act(fin->X, fin->ldx, fin->smooth, M, K, const_cast<int8_t*>(Xq),
                                                       const_cast<float*>(sa),
                                                       reinterpret_cast<quasar_stream_t>(stream));
    if (sq != QUASAR_OK) return sq;
    p.X = nullptr;
    e = go();
  }
  if (e == cudaErrorInvalidValue) return QUASAR_ERR_UNSUPPORTED;
  return cuda_status(e);
}

}  // namespace skinny
}  // namespace quasar
