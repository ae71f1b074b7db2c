// A3 + A4 for a few tokens (M <= 16): the W8A8 verify linear on the
// register tensor path.
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
// tcgen05.mma of M = 128, K = 16 takes ~50 cycles whatever N <= 64 is (it is
// bound by its own operand traffic), i.e. ~41 weight bytes per cycle before
// the weights are even widened into TMEM.  The warp-level m16n8k16 fp16 MMA
// runs at ~2048 flop/clk/SM on sm_103a and takes its weight operand straight
// from registers: at M <= 8 it covers 128 weight bytes per cycle, at M = 32
// still 32, against the ~22 bytes per cycle an SM must stream for HBM-rate.
// So for M <= 32 the weights go HBM -> shared memory (1-D bulk copies, the
// same packed blocks the tcgen05 kernel reads) -> registers (ldmatrix) ->
// fp16 (exact) -> mma.sync, with fp32 accumulators that stay exact integers
// (see RUN_BLOCKS), and the tcgen05 kernel keeps the larger M.
//
// Work split.  Persistent grid, one CTA per SM, each CTA streaming an equal
// contiguous range of (weight tile, 128-K block) items (stream-K).  Inside a
// block, consumer warp (kq, rg) owns K bytes [32 kq, 32 kq + 32) of weight
// rows [64 rg, 64 rg + 64): 4 row tiles x 2 K steps x NT/8 token tiles of
// MMAs.  Owning K rather than rows means each warp widens only its own token
// columns, so the token operand is converted twice per block instead of
// eight times; the four K owners of a row tile are summed through shared
// memory once per accumulation run.
//
// Schedules.  A split tile's sums must cross CTAs, and doing that at the end
// of a launch puts a chain of dependent memory round trips after the last
// weight byte, so the exchange is kept off the launch's tail:
//  * few tiles (2 x tiles <= SMs): a thread-block cluster of C CTAs takes one
//    tile, each CTA a 1/C slice of its K blocks; the slices are summed
//    through distributed shared memory between two cluster barriers.
//  * otherwise: the tiles that do not divide evenly over the CTAs are split
//    stream-K over all CTAs and done first; each CTA then streams whole
//    tiles.  A split tile is summed without atomics on the data: each
//    contributor stores its integer partial sums into a slot of its own in
//    the workspace and counts its K blocks on a per-(tile, warp) counter; the
//    warp that completes the count adds up the slots of every contributor and
//    runs the epilogue, while the whole tiles still stream.
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

constexpr int BM = 128;           // weight rows per tile
constexpr int BK = 128;           // K bytes per block
constexpr int BLOCK_BYTES = BM * BK;
constexpr int KQ = 4;             // K quarters (32 K = 2 MMA K steps each)
constexpr int RG = 2;             // row groups (64 rows = 4 row tiles each)
constexpr int CWARPS = KQ * RG;   // consumer warps; warp w finalizes row tile w
constexpr int CNT_STRIDE = 16;    // counters per tile in the shared workspace layout
constexpr int PRODUCER_WARP = CWARPS;
constexpr int THREADS = 32 * (CWARPS + 1);
constexpr int RED_BAR = 1;        // named barrier of the consumer warps
constexpr int MAX_CTAS = 160;     // grid cap; sizes the partial-sum slots
// A warp adds 32 products per block into each fp32 accumulator, each product
// at most 127^2 = 16129 in magnitude: 32 blocks x 32 x 16129 < 2^24, so over
// a run of <= 32 blocks every partial sum is an exact integer in fp32.
constexpr int RUN_BLOCKS = 32;

template <int NT8>
struct Cfg {
  static constexpr int NT = 8 * NT8;                        // token columns (padded to 8)
  static constexpr int XB = NT * BK;                        // INT8 token tile of a block
  static constexpr int STAGE = BLOCK_BYTES + XB;            // multiple of 1024 (swizzle atoms)
  static constexpr int RED = 8 * KQ * NT8 * 32 * 16;        // fp32 partials: [row tile][kq][token tile][lane]
  static constexpr int FIN = 8 * NT8 * 32 * 16;             // int32 run sums: [row tile][token tile][lane]
  static constexpr int SLOT = 8 * NT8 * 32;                 // int4 per partial-sum slot (128 rows x NT)
  static constexpr int SCL = (32 + 2 * BM) * 4;             // staged scales: sa[32], sw of 2 tiles
  static constexpr int S_FIT = (225 * 1024 - RED - FIN - SCL - 1024 - 256) / STAGE;
  static constexpr int S = S_FIT < 12 ? S_FIT : 12;         // stages in flight
  static constexpr int SMEM = 1024 + S * STAGE + RED + FIN + SCL + 256;
  static_assert(STAGE % 1024 == 0, "stage alignment");
  static_assert(S >= 4, "pipeline depth");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Params {
  const uint8_t* wp;  // packed weights, [n_tiles][KB][128 rows][128 B]
  const float* sa;
  const float* sw;
  int M, N, K;
  int KB;           // K blocks per tile
  int mode;         // 0: split tiles stream-K, then whole tiles; 1: cluster per tile
  int csize;        // mode 1: CTAs per cluster (K slices per tile)
  int split_tiles;  // mode 0: tiles [0, split_tiles) are split stream-K ...
  int total1;       //   ... over their split_tiles * KB blocks
  int whole_per;    // mode 0: whole tiles per CTA, after the split tiles
  __nv_bfloat16* Y;
  int ldy;
  int32_t* acc_out;   // int32 mode when non-null
  int4* slots;        // [grid][2] partial sums, each [row tile][token tile][lane] int4
  uint32_t* ws_cnt;   // [n_tiles][16] K-block counters per finalizer warp (8 used), zero between calls
  unsigned int* err;
  unsigned long long limit_ns;
};

// One CTA's work: split items [s0, s1) (item i = K block i % KB of tile
// i / KB), then whole tiles [w0, w1).
struct Sched {
  int s0, s1, w0, w1;
};

QUASAR_DEVICE_INLINE int range_begin(int c, int total, int grid);

QUASAR_DEVICE_INLINE Sched schedule_of(int c, int grid, int KB, int mode, int csize, int split_tiles, int total1,
                                       int whole_per) {
  Sched sc;
  if (mode == 1) {
    const int t = c / csize, q = c % csize;
    sc.s0 = t * KB + (q * KB) / csize;
    sc.s1 = t * KB + ((q + 1) * KB) / csize;
    sc.w0 = sc.w1 = 0;
  } else {
    sc.s0 = range_begin(c, total1, grid);
    sc.s1 = range_begin(c + 1, total1, grid);
    sc.w0 = split_tiles + c * whole_per;
    sc.w1 = sc.w0 + whole_per;
  }
  return sc;
}

// Walks a schedule one K block per step.  Segments (the CTA's blocks of one
// tile within a phase) and accumulation runs (<= RUN_BLOCKS blocks of a
// segment) are contiguous.
struct Walk {
  int t, kb, kb_first, left, left2, w_next, phase;
  __device__ Walk(const Sched& sc, int KB) {
    if (sc.s1 > sc.s0) {
      phase = 1;
      t = sc.s0 / KB;
      kb = kb_first = sc.s0 % KB;
      left = sc.s1 - sc.s0;
      left2 = (sc.w1 - sc.w0) * KB;
    } else {
      phase = 2;
      t = sc.w0;
      kb = kb_first = 0;
      left = (sc.w1 - sc.w0) * KB;
      left2 = 0;
    }
    w_next = sc.w0;
  }
  __device__ bool more() const { return left > 0; }
  __device__ bool seg_last(int KB) const { return left == 1 || kb + 1 == KB; }
  __device__ bool run_last(int KB) const { return seg_last(KB) || ((kb - kb_first + 1) % RUN_BLOCKS) == 0; }
  __device__ void next(int KB) {
    --left;
    if (++kb == KB) {
      kb = 0;
      kb_first = 0;
      ++t;
    }
    if (left == 0 && left2 > 0) {   // enter the whole tiles
      phase = 2;
      t = w_next;
      kb = kb_first = 0;
      left = left2;
      left2 = 0;
    }
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

// Cluster-wide barrier of every thread of every CTA in the cluster (release
// on arrive, acquire on wait); warp-converged callers only.
QUASAR_DEVICE_INLINE void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// int4 at the same shared-memory offset in cluster CTA `rank`.
QUASAR_DEVICE_INLINE int4 ld_dsmem_int4(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
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

// A finalizer warp's share of a tile is row tile mt, all token tiles: lane
// holds int4 v[ni] per token tile ni, whose element j is row 8 (j >> 1) + g
// of the row tile, token 8 ni + 2c + (j & 1).  `sa_s` holds sa of every
// token (shared memory), `swt` sw of the tile's 128 rows (shared memory for
// the CTA's first and last tile, else global).
template <int NT8>
QUASAR_DEVICE_INLINE void epilogue(const Params& p, const int4 (&v4)[NT8], int t, int mt, int lane,
                                   const float* sa_s, const float* swt) {
  const int g = lane >> 2, c = lane & 3;
  const int nrow0 = t * BM + mt * 16 + g;
  float swr[2] = {0.f, 0.f};
  if (!p.acc_out) {
    swr[0] = swt[mt * 16 + g];
    swr[1] = swt[mt * 16 + g + 8];
  }
#pragma unroll
  for (int ni = 0; ni < NT8; ++ni) {
    const int32_t v[4] = {v4[ni].x, v4[ni].y, v4[ni].z, v4[ni].w};
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

// Contributors of split tile t and the slot each used: a contributor's
// segment of a split tile is its first segment (slot 0) or its last (slot
// 1); every one is partial.
template <int NT8>
QUASAR_DEVICE_INLINE int4* slot_ptr(const Params& p, int cc, int t, int mt, int lane, int grid) {
  const int first_t = range_begin(cc, p.total1, grid) / p.KB;
  return p.slots + ((size_t)cc * 2 + (first_t == t ? 0 : 1)) * Cfg<NT8>::SLOT + (size_t)mt * NT8 * 32 + lane;
}

// Sum of every contributor's slot for this warp's share of split tile t
// (loads only: four contributors in flight at a time).
template <int NT8>
QUASAR_DEVICE_INLINE void load_slots(const Params& p, int t, int mt, int lane, int grid, int4 (&s)[NT8]) {
  const int c_lo = cta_of_block(t * p.KB, p.total1, grid);
  const int c_hi = cta_of_block((t + 1) * p.KB - 1, p.total1, grid);
#pragma unroll
  for (int ni = 0; ni < NT8; ++ni) s[ni] = make_int4(0, 0, 0, 0);
  for (int c0 = c_lo; c0 <= c_hi; c0 += 4) {
    int4 v[4][NT8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni)
        v[u][ni] = (c0 + u <= c_hi) ? __ldcg(slot_ptr<NT8>(p, c0 + u, t, mt, lane, grid) + ni * 32)
                                    : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni) {
        s[ni].x += v[u][ni].x;
        s[ni].y += v[u][ni].y;
        s[ni].z += v[u][ni].z;
        s[ni].w += v[u][ni].w;
      }
  }
}

// Each slot share is read exactly once (by the warp that completes the tile)
// and zeroed after the read, so the workspace is left as it was found.
template <int NT8>
QUASAR_DEVICE_INLINE void zero_slots(const Params& p, int t, int mt, int lane, int grid) {
  const int c_lo = cta_of_block(t * p.KB, p.total1, grid);
  const int c_hi = cta_of_block((t + 1) * p.KB - 1, p.total1, grid);
  for (int cc = c_lo; cc <= c_hi; ++cc) {
    int4* slot = slot_ptr<NT8>(p, cc, t, mt, lane, grid);
#pragma unroll
    for (int ni = 0; ni < NT8; ++ni) __stcg(slot + ni * 32, make_int4(0, 0, 0, 0));
  }
}

// Publish partial segments: one fence for this warp's slot stores, then the
// K-block count of each segment (tile ta with na blocks, and tile tb with nb
// blocks when tb >= 0); a warp whose count completes a tile sums the tile's
// slots and runs its epilogue.  Both tiles' slots are loaded before either
// epilogue so that their latencies overlap.
template <int NT8>
QUASAR_DEVICE_INLINE void count_segments(const Params& p, int ta, int na, int tb, int nb, int mt, int lane,
                                         int grid, const float* sa_s, const float* swa, const float* swb) {
  __threadfence();
  __syncwarp();
  uint32_t last_mask = 0;
  if (lane == 0) {
    const uint32_t old_a = atomicAdd(&p.ws_cnt[(size_t)ta * CNT_STRIDE + mt], (uint32_t)na);
    const uint32_t old_b = (tb >= 0) ? atomicAdd(&p.ws_cnt[(size_t)tb * CNT_STRIDE + mt], (uint32_t)nb) : 0u;
    if (old_a + (uint32_t)na == (uint32_t)p.KB) last_mask |= 1u;
    if (tb >= 0 && old_b + (uint32_t)nb == (uint32_t)p.KB) last_mask |= 2u;
  }
  last_mask = __shfl_sync(0xffffffffu, last_mask, 0);
  if (!last_mask) return;
  __threadfence();
  int4 va[NT8], vb[NT8];
  if (last_mask & 1u) load_slots<NT8>(p, ta, mt, lane, grid, va);
  if (last_mask & 2u) load_slots<NT8>(p, tb, mt, lane, grid, vb);
  if (last_mask & 1u) {
    zero_slots<NT8>(p, ta, mt, lane, grid);
    epilogue<NT8>(p, va, ta, mt, lane, sa_s, swa);
    if (lane == 0) p.ws_cnt[(size_t)ta * CNT_STRIDE + mt] = 0u;   // ready for the next call
  }
  if (last_mask & 2u) {
    zero_slots<NT8>(p, tb, mt, lane, grid);
    epilogue<NT8>(p, vb, tb, mt, lane, sa_s, swb);
    if (lane == 0) p.ws_cnt[(size_t)tb * CNT_STRIDE + mt] = 0u;
  }
}

template <int NT8>
__global__ void __launch_bounds__(THREADS, 1)
w8a8_skinny_kernel(const __grid_constant__ CUtensorMap tmX, const Params p) {
  using C = Cfg<NT8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;                                     // S x [W 16 KB | X NT x 128 B]
  float4* red = reinterpret_cast<float4*>(smem + C::S * C::STAGE);
  int4* fin = reinterpret_cast<int4*>(smem + C::S * C::STAGE + C::RED);
  float* sa_s = reinterpret_cast<float*>(smem + C::S * C::STAGE + C::RED + C::FIN);   // [32]
  float* sw_s = sa_s + 32;                                                                // [2][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::S * C::STAGE + C::RED + C::FIN + C::SCL);
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
  const Sched sc = schedule_of((int)blockIdx.x, grid, KB, p.mode, p.csize, p.split_tiles, p.total1, p.whole_per);

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      // Weights do not depend on the previous kernel: fill every stage first.
      int pre = 0;
      {
        Walk w(sc, KB);
        for (; pre < C::S && w.more(); ++pre, w.next(KB)) {
          mbar_arrive_expect_tx(&full[pre], (uint32_t)C::STAGE);
          bulk_load(stages + pre * C::STAGE, p.wp + ((size_t)w.t * KB + w.kb) * BLOCK_BYTES, BLOCK_BYTES,
                    &full[pre], pol_w);
        }
      }
      pdl_wait();  // token codes come from the previous kernel
      Walk w(sc, KB);
      Ring<C::S> rg;
      int issued = 0;
      for (; w.more(); w.next(KB), rg.next(), ++issued) {
        uint8_t* st = stages + rg.s * C::STAGE;
        if (issued >= pre) {
          if (!mbar_wait(&empty[rg.s], rg.ph ^ 1u, abort_flag, p.err, SITE_SKINNY_EMPTY, p.limit_ns)) break;
          mbar_arrive_expect_tx(&full[rg.s], (uint32_t)C::STAGE);
          bulk_load(st, p.wp + ((size_t)w.t * KB + w.kb) * BLOCK_BYTES, BLOCK_BYTES, &full[rg.s], pol_w);
        }
        tma_load_2d(st + BLOCK_BYTES, &tmX, w.kb * BK, 0, &full[rg.s], pol_x);
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
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int kq = warp & (KQ - 1);   // K bytes [32 kq, 32 kq + 32) of each block
  const int rg = warp / KQ;         // rows [64 rg, 64 rg + 64): row tiles 4 rg .. 4 rg + 3
  const int g = lane >> 2, c = lane & 3;
  const int mt_f = warp;            // the row tile this warp finalizes
  pdl_wait();                       // scales and workspace belong to the previous kernel until here
  const int t_first = (sc.s1 > sc.s0) ? sc.s0 / KB : sc.w0;
  const int t_last = (sc.w1 > sc.w0) ? sc.w1 - 1 : (sc.s1 - 1) / KB;
  const int t_first1 = sc.s0 / KB;  // first tile of the split range (its slot 0)
  // Stage the dequantization scales the epilogues will need: every token's
  // sa, and sw of the first and last tile of this CTA (read after the first
  // run-end barrier, which orders these stores).
  if (!p.acc_out) {
    for (int i = threadIdx.x; i < 32 + 2 * BM; i += CWARPS * 32) {
      if (i < 32) {
        sa_s[i] = (i < p.M) ? __ldg(&p.sa[i]) : 0.f;
      } else {
        const int r = i - 32;
        const int n = (r < BM ? t_first : t_last) * BM + (r & (BM - 1));
        sw_s[r] = (n < p.N) ? __ldg(&p.sw[n]) : 0.f;
      }
    }
  }

  float acc[4][NT8][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int n = 0; n < NT8; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][n][j] = 0.f;
  // Finished integer sums of this warp's row tile, kept in shared memory
  // (touched once per run).
  int4* share = fin + mt_f * NT8 * 32 + lane;
#pragma unroll
  for (int ni = 0; ni < NT8; ++ni) share[ni * 32] = make_int4(0, 0, 0, 0);

  // Per-lane address parts.  ldmatrix over one K step of 32 rows: lanes
  // 8i..8i+7 give rows 8i..8i+7, i.e. matrix i = (row tile i >> 1, row half
  // i & 1).  The second K step's chunk differs from the first in bit 0 only,
  // i.e. its offset is the first one's ^ 16.
  const uint32_t a_off = (uint32_t)((rg * 64 + lane) * BK + (((2 * kq) ^ (lane & 7)) << 4));
  const uint32_t b_off = (uint32_t)(BLOCK_BYTES + g * BK + (((2 * kq) ^ g) << 4) + 4 * c);
  const uint32_t stages_u32 = smem_u32(stages);

  bool bad = false;
  // Partial segments of the split range (at most two: its first and last)
  // are counted together when the range ends, so that one fence covers both.
  int seg_ta = -1, seg_na = 0, seg_tb = -1, seg_nb = 0;
  // sw of tile t: staged for the CTA's first and last tile.
  auto sw_of = [&](int t) -> const float* {
    return t == t_first ? sw_s : t == t_last ? sw_s + BM : p.sw + (size_t)t * BM;
  };
  Walk w(sc, KB);
  Ring<C::S> r;
  for (; w.more(); w.next(KB), r.next()) {
    if (!bad) {
      const bool ok = mbar_wait(&full[r.s], r.ph, abort_flag, p.err, SITE_SKINNY_FULL, p.limit_ns);
      bad = !__all_sync(0xffffffffu, ok);
    }
    if (!bad) {
      const uint32_t st = stages_u32 + (uint32_t)(r.s * C::STAGE);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        // Token operands (row n = 8 ni + g of the swizzled tile sits at
        // n * 128, chunk ch at (ch ^ (n & 7)) * 16).
        uint32_t bq[NT8][2];
#pragma unroll
        for (int ni = 0; ni < NT8; ++ni)
          s8x4_to_f16x4(lds32(st + (b_off ^ (ks << 4)) + (uint32_t)(ni * 8 * BK)), bq[ni][0], bq[ni][1]);
#pragma unroll
        for (int i2 = 0; i2 < 2; ++i2) {
          uint32_t d[4];
          ldsm_x4(st + (a_off ^ (ks << 4)) + (uint32_t)(i2 * 32 * BK), d[0], d[1], d[2], d[3]);
#pragma unroll
          for (int ii = 0; ii < 2; ++ii) {
            uint32_t a0, a1, a2, a3;
            u8x4_to_f16x4(d[2 * ii], a0, a2);       // rows g: K slots 2c.. (bytes 4c, 4c+1), 2c+8.. (4c+2, 4c+3)
            u8x4_to_f16x4(d[2 * ii + 1], a1, a3);   // rows g + 8
#pragma unroll
            for (int ni = 0; ni < NT8; ++ni)
              mma_16816(acc[2 * i2 + ii][ni], a0, a1, a2, a3, bq[ni][0], bq[ni][1]);
          }
        }
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
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni) {
        red[(((4 * rg + i) * KQ + kq) * NT8 + ni) * 32 + lane] =
            make_float4(acc[i][ni][0], acc[i][ni][1], acc[i][ni][2], acc[i][ni][3]);
        acc[i][ni][0] = acc[i][ni][1] = acc[i][ni][2] = acc[i][ni][3] = 0.f;
      }
    named_barrier_or(RED_BAR, CWARPS * 32, 0u);
#pragma unroll
    for (int ni = 0; ni < NT8; ++ni) {
      int4 f = share[ni * 32];
#pragma unroll
      for (int q = 0; q < KQ; ++q) {
        const float4 v = red[((mt_f * KQ + q) * NT8 + ni) * 32 + lane];
        f.x += __float2int_rn(v.x);
        f.y += __float2int_rn(v.y);
        f.z += __float2int_rn(v.z);
        f.w += __float2int_rn(v.w);
      }
      share[ni * 32] = f;
    }
    if (!w.seg_last(KB)) continue;

    // ---- end of this CTA's segment of tile t.
    const int t = w.t;
    const int nb = w.kb - w.kb_first + 1;
    if (p.mode == 1) break;   // the only segment: summed across the cluster below
    if (nb == KB) {
      int4 v[NT8];
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni) v[ni] = share[ni * 32];
      epilogue<NT8>(p, v, t, mt_f, lane, sa_s, sw_of(t));   // the whole tile
    } else {
      // Partial segment of the split range: store the share into this CTA's
      // slot for it (0 = the range's first segment, 1 = its last).
      int4* slot = p.slots + ((size_t)blockIdx.x * 2 + (t == t_first1 ? 0 : 1)) * C::SLOT +
                   (size_t)mt_f * NT8 * 32 + lane;
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni) slot[ni * 32] = share[ni * 32];
      if (seg_ta < 0) {
        seg_ta = t;
        seg_na = nb;
      } else {
        seg_tb = t;
        seg_nb = nb;
      }
    }
    if (w.phase == 1 && w.left == 1 && seg_ta >= 0) {
      // The split range ends here: publish its partial segments now, while
      // the whole tiles (if any) still stream.
      count_segments<NT8>(p, seg_ta, seg_na, seg_tb, seg_nb, mt_f, lane, grid, sa_s, sw_of(seg_ta),
                          seg_tb >= 0 ? sw_of(seg_tb) : sw_s);
      seg_ta = -1;
    }
#pragma unroll
    for (int ni = 0; ni < NT8; ++ni) share[ni * 32] = make_int4(0, 0, 0, 0);
  }

  if (p.mode == 1) {
    // Cluster split: every CTA of the cluster holds the sums of one K slice of
    // tile t in `fin`.  After the barrier each row tile is finished by one
    // CTA (row tile mt in the CTA of rank mt % C), reading the other slices
    // through distributed shared memory; the second barrier keeps every CTA's
    // shared memory alive until those reads are done.
    __syncwarp();
    cluster_sync_all();
    const int csz = p.csize;
    const int rank = (int)blockIdx.x % csz;
    if (!bad && (mt_f % csz) == rank) {
      int4 v[NT8];
#pragma unroll
      for (int ni = 0; ni < NT8; ++ni) v[ni] = share[ni * 32];
      for (int q = 0; q < csz; ++q) {
        if (q == rank) continue;
#pragma unroll
        for (int ni = 0; ni < NT8; ++ni) {
          const int4 u = ld_dsmem_int4(share + ni * 32, (uint32_t)q);
          v[ni].x += u.x;
          v[ni].y += u.y;
          v[ni].z += u.z;
          v[ni].w += u.w;
        }
      }
      epilogue<NT8>(p, v, t_first, mt_f, lane, sa_s, sw_s);
    }
    __syncwarp();
    cluster_sync_all();
  }
}

// ------------------------------------------------------------------ host side

template <int NT8>
static cudaError_t configure(int dev) {
  static int configured[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(w8a8_skinny_kernel<NT8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<NT8>::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return cudaSuccess;
}

template <int NT8>
static cudaLaunchConfig_t config_of(int grid, int csize, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg<NT8>::SMEM;
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

// Clusters of `csize` CTAs of this kernel that the device keeps resident at
// once (0 if unknown); cached per device and cluster size.
template <int NT8>
static int resident_clusters(int dev, int csize) {
  static int cache[64][9];
  static bool init[64][9] = {};
  if (dev < 0 || dev >= 64 || csize < 2 || csize > 8) return 0;
  if (!init[dev][csize]) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = config_of<NT8>(csize * 16, csize, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, w8a8_skinny_kernel<NT8>, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();
    }
    cache[dev][csize] = n;
    init[dev][csize] = true;
  }
  return cache[dev][csize];
}

template <int NT8>
static cudaError_t launch(const CUtensorMap& tx, Params p, int sms, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = configure<NT8>(dev);
  if (e != cudaSuccess) return e;
  const int n_tiles = (p.N + BM - 1) / BM;
  // Few tiles: one cluster per tile, as many K slices as fit in one wave.
  int csize = std::min(std::min(8, sms / n_tiles), p.KB);
  while (csize >= 2 && resident_clusters<NT8>(dev, csize) < n_tiles) --csize;
  int grid;
  if (csize >= 2) {
    p.mode = 1;
    p.csize = csize;
    p.split_tiles = 0;
    p.total1 = 0;
    p.whole_per = 0;
    grid = n_tiles * csize;
  } else {
    p.mode = 0;
    p.csize = 1;
    grid = std::min(sms, MAX_CTAS);
    p.whole_per = n_tiles / grid;
    p.split_tiles = n_tiles - p.whole_per * grid;
    p.total1 = p.split_tiles * p.KB;
    if (p.whole_per == 0) grid = std::min(grid, p.total1);
    if ((unsigned long long)(p.total1 + 1) * (unsigned long long)(grid + 1) >= (1ull << 32))
      return cudaErrorInvalidValue;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = config_of<NT8>(grid, p.csize, stream, attr);
  return cudaLaunchKernelEx(&cfg, w8a8_skinny_kernel<NT8>, tx, p);
}

bool handles(int M) { return M >= 1 && M <= 16; }

// Partial-sum slots this kernel may need after the counters: two per CTA.
// Like the counters they are zero between calls (each is zeroed by its
// reader).
size_t slots_bytes(int M, int N, int K) {
  if (!handles(M) || N <= 0 || K <= 0) return 0;
  const long long total = (long long)((N + BM - 1) / BM) * ((K + BK - 1) / BK);
  const long long ctas = std::min<long long>(total, MAX_CTAS);
  return (size_t)ctas * 2 * (size_t)BM * 8 * ((M + 7) / 8) * 4;
}

// Arguments were validated by the caller; ws_cnt holds >= n_tiles * 16
// zeroed counters, `slots` slots_bytes() bytes (no initial value needed).
quasar_status_t run(const int8_t* Xq, const float* sa, const int8_t* Wp, const float* sw, int M, int N, int K,
                    void* Y, int ldy, int32_t* acc_out, uint32_t* ws_cnt, void* slots, cudaStream_t stream) {
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
  if (!p.err) return QUASAR_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return QUASAR_ERR_CUDA;
  cudaError_t e;
  switch (nt8) {
    case 1: e = launch<1>(tx, p, sms, stream); break;
    default: e = launch<2>(tx, p, sms, stream); break;   // handles() keeps M <= 16
  }
  if (e == cudaErrorInvalidValue) return QUASAR_ERR_UNSUPPORTED;
  return cuda_status(e);
}

}  // namespace skinny
}  // namespace quasar
