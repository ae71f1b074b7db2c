// The verifier's BF16 lm_head with the verification reductions in its
// epilogue (the logits are never written).
//
// Quasar summary nl §2 "Methodologie" / ko §2 "방법론": the verifier keeps its
// logits in high precision (the last matmul stays BF16) and checks the drafts
// on them with greedy or rejection acceptance.  Per token row those tests need
// only the argmax, the maximum, the sum of exp((l - max) / T) and the draft's
// own logit, so this file computes
//     l[c][v] = bf16_rne( fp32 sum_k H[c][k] * W[v][k] )
// on the tensor cores and reduces every 128-row vocabulary tile of it to one
// record per token row, instead of writing the [rows][V] logits tensor.
//
// lm_head_kernel: persistent, one CTA per SM, vocabulary tiles dealt round
// robin.  Swap-AB: 128 vocabulary rows are the MMA's M (the A operand, from
// the weight stream), the token rows its N (B, at most 256 per MMA, two MMAs
// for more).  The weight is packed offline into contiguous 16 KB blocks of
// 128 rows x 64 K values, each already in the 128B-swizzled K-major layout
// the MMA reads, and streams in with 1-D bulk copies: whole blocks keep the
// HBM accesses long and sequential, where a 2-D tile of a row-major [V][K]
// weight would read 128 bytes from each of 128 rows 8 KB apart.  The token
// rows come by TMA (they are small and stay in L2).  tcgen05.mma kind::f16
// with BF16 inputs accumulates in fp32 in TMEM.  Roles: warps 0-3 drain the
// accumulator (TMEM lane quarter = warp), warp 4 issues the copies, warp 5
// the MMAs, warp 6 does every mbarrier wait for warp 5 (an MMA-issuing
// thread that touches memory waits for its queued MMAs to be accepted, which
// would drain the tensor pipe at every stage).
//
// The accumulator of local tile i sits at TMEM column 0 (i even) or
// 512 - Tp (i odd).  For Tp <= 256 the two regions are disjoint, so the
// drain of tile i overlaps all of tile i+1's MMAs; above 256 they share
// columns [512 - Tp, Tp), which the drain reads first and then releases.
//
// Epilogue per tile and token column: each lane holds one vocabulary row;
// the warp reduces 32 columns x 32 rows with a transposing butterfly (after
// five exchange steps lane l holds column l's result, 31 shuffles per 32
// columns).  The argmax travels as one 32-bit key: the BF16 logit in an
// order-preserving 16-bit form above 0xFFFF minus the row within the tile,
// so the larger key is the larger logit and, on ties, the lower index.
//
// lm_head_finalize_kernel: one CTA per token row merges that row's tile
// records in tile order (deterministic), and the last row of a sequence to
// finish applies the acceptance rule of quasar_verify_accept.  Every value
// it reads from the workspace it zeroes again, so a call leaves the
// workspace zero-filled like every other call of the library.
#include <climits>

#include "quasar_common.cuh"

namespace quasar {
namespace lmhead {

constexpr int BMV = 128;            // vocabulary rows per tile (MMA M)
constexpr int BKE = 64;             // K elements per stage (one 128-byte swizzle row)
constexpr int A_BYTES = BMV * 128;  // 16 KB of weights per stage (one packed block)
constexpr int EPI_WARPS = 4;       // warps 0-3: accumulator drain (TMEM lane quarter = warp)
constexpr int PRODUCER_WARP = 4;
constexpr int MMA_WARP = 5;
constexpr int WAITER_WARP = 6;
constexpr int THREADS = 32 * 7;
constexpr int MMA_BAR_ID = 1;       // MMA + waiter warps
constexpr int EPI_BAR_ID = 2;       // the four epilogue warps
constexpr int TMEM_COLS = 512;
constexpr int MAX_ROWS = 512;       // token rows per call (TMEM columns)
constexpr int MAX_STAGES = 8;
constexpr int SMEM_LIMIT = 232448;

// MODE_SAMPLE_NEXT is a finishing mode only: the matmul runs as MODE_SAMPLED.
enum Mode : int { MODE_LOGITS = 0, MODE_GREEDY = 1, MODE_SAMPLED = 2, MODE_SAMPLE_NEXT = 3 };

struct Params {
  int Mt;          // token rows (B * (D + 1) for verification)
  int Tp;          // token rows padded to 32
  int nmma;        // MMAs per K step (1 or 2)
  int Nh;          // token rows per MMA (Tp / nmma)
  int V, K;
  int n_vt;        // vocabulary tiles
  int KB;          // K steps of 64
  int stages;
  uint32_t idesc;
  const uint8_t* wp;      // packed weight blocks [n_vt][KB][16 KB]
  __nv_bfloat16* logits;  // MODE_LOGITS: [Mt][ldl]
  long long ldl;
  uint2* rec;      // [Mt][n_vt] {key, fp32 bits of the tile's exp-sum}
  float* dl;       // [Mt] the draft's logit (MODE_SAMPLED)
  const int32_t* draft;   // [B][D]
  int D;
  float k2;        // log2(e) / T
  unsigned int* err;
  unsigned long long limit_ns;
};

__host__ __device__ constexpr uint32_t stage_bytes(int Tp) { return (uint32_t)A_BYTES + (uint32_t)Tp * 128u; }

// Dynamic shared memory: alignment slack, the stage ring, the per-quarter
// partial results, the draft of every token column, barriers.
__host__ __device__ constexpr uint32_t smem_bytes(int Tp, int stages) {
  return 1024u + (uint32_t)stages * stage_bytes(Tp) + 32u * (uint32_t)Tp + 4u * (uint32_t)Tp + 256u;
}

// Shared-memory matrix descriptor of a 128B-swizzled K-major tile whose
// 8-row groups are 1024 bytes apart (start >> 4 in bits 0-13, leading offset
// 1 (unused when swizzled) in 16-29, stride offset 1024 >> 4 in 32-45,
// version 1 at bit 46, swizzle mode 2 = 128 B in bits 61-63).
QUASAR_DEVICE_INLINE uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// The four K=16 MMAs of one 64-K stage for one token block, both operands
// from shared memory, issued from one asm statement so that nothing is
// scheduled between them.  Descriptor starts advance 32 bytes (2 units of
// 16) per K step inside the 128-byte swizzle row.
QUASAR_DEVICE_INLINE void mma_stage(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, t;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc0), "l"(a + 2), "l"(b + 2), "l"(a + 4), "l"(b + 4), "l"(a + 6),
      "l"(b + 6)
      : "memory");
}

QUASAR_DEVICE_INLINE void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// BF16 bits <-> a 16-bit key whose unsigned order is the numeric order.
QUASAR_DEVICE_INLINE uint32_t ord16(uint32_t b) { return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u); }
QUASAR_DEVICE_INLINE float key_value(uint32_t key) {
  const uint32_t k = key >> 16;
  const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  return __uint_as_float(b << 16);
}

struct MaxOp {
  QUASAR_DEVICE_INLINE uint32_t operator()(uint32_t a, uint32_t b) const { return a > b ? a : b; }
};
struct AddOp {
  QUASAR_DEVICE_INLINE float operator()(float a, float b) const { return a + b; }
};

// Reduces v[i] over the warp's 32 lanes for 32 columns i at once: at the
// step of offset o, a lane keeps the half of its columns selected by its bit
// o, sends the other half to lane ^ o and combines.  Afterwards lane l holds
// column l's result.
template <class T, class Op>
QUASAR_DEVICE_INLINE T transpose_reduce32(T (&v)[32], int lane, Op op) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const T send = up ? v[i] : v[i + o];
      const T keep = up ? v[i + o] : v[i];
      const T recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = op(keep, recv);
    }
  }
  return v[0];
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tmH, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  const int Tp = p.Tp;
  const uint32_t STAGE = stage_bytes(Tp);
  uint8_t* ring = smem;                                               // S x [A 16 KB | B Tp x 128 B]
  uint2* part = reinterpret_cast<uint2*>(smem + (size_t)S * STAGE);   // [4][Tp]
  int* sdraft = reinterpret_cast<int*>(part + 4 * Tp);                // [Tp]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sdraft + Tp);
  uint64_t* full = bars;                 // [S] copies landed
  uint64_t* empty = full + S;            // [S] MMAs done reading
  uint64_t* acc_full = empty + S;        // a tile's MMAs are complete
  uint64_t* acc_free = acc_full + 1;     // the drain released the shared columns
  uint64_t* mma_done = acc_free + 1;     // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_free, EPI_WARPS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    prefetch_tmap(&tmH);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int KB = p.KB;
  const int my_tiles = (p.n_vt - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int items = my_tiles * KB;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      // The weights do not depend on earlier kernels: the first S stages'
      // weight copies start before waiting for the previous kernel.
      const int pre = items < S ? items : S;
      for (int i = 0; i < pre; ++i) {
        const int t = (int)blockIdx.x + (i / KB) * (int)gridDim.x;
        mbar_arrive_expect_tx(&full[i], STAGE);
        bulk_load(ring + (size_t)i * STAGE, p.wp + ((size_t)t * KB + i % KB) * A_BYTES, A_BYTES, &full[i], pol_w);
      }
      pdl_wait();  // H is written by the previous kernel
      int issued = 0;
      for (int i = 0; i < items; ++i, ++issued) {
        const int s = i % S;
        const uint32_t ph = (uint32_t)(i / S) & 1u;
        const int t = (int)blockIdx.x + (i / KB) * (int)gridDim.x;
        const int kb = i % KB;
        uint8_t* st = ring + (size_t)s * STAGE;
        if (i >= pre) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.err, SITE_LMH_EMPTY, p.limit_ns)) break;
          mbar_arrive_expect_tx(&full[s], STAGE);
          bulk_load(st, p.wp + ((size_t)t * KB + kb) * A_BYTES, A_BYTES, &full[s], pol_w);
        }
        for (int h = 0; h < p.nmma; ++h)
          tma_load_2d(st + A_BYTES + (size_t)h * p.Nh * 128, &tmH, kb * BKE, h * p.Nh, &full[s], pol_h);
      }
      // Never leave with copies in flight: wait for the last phase issued on
      // every stage (already complete in a normal run).
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / S) * S;
        volatile int dummy = 0;
        mbar_wait(&full[s], (uint32_t)(last / S) & 1u, &dummy, p.err, SITE_LMH_DRAIN, p.limit_ns);
      }
    }
  } else if (warp == MMA_WARP || warp == WAITER_WARP) {
    const uint64_t ring_desc = sw128_desc(smem_u32(ring));
    int issued = 0;
    for (int i = 0; i < items; ++i) {
      const int s = i % S;
      const uint32_t ph = (uint32_t)(i / S) & 1u;
      const int lt = i / KB;  // local tile
      const int kb = i % KB;
      uint32_t abort_in = 0;
      if (warp == WAITER_WARP) {
        bool ok = true;
        if (kb == 0 && lt >= 1)
          ok = mbar_wait(acc_free, (uint32_t)(lt - 1) & 1u, abort_flag, p.err, SITE_LMH_ACCFREE, p.limit_ns);
        ok = ok && mbar_wait(&full[s], ph, abort_flag, p.err, SITE_LMH_FULL, p.limit_ns);
        abort_in = __all_sync(0xffffffffu, ok) ? 0u : 1u;
      }
      if (named_barrier_or(MMA_BAR_ID, 64, abort_in)) break;
      if (warp == MMA_WARP) {
        if (lane == 0) {
          tc_fence_after();
          const uint32_t base = (lt & 1) ? (uint32_t)(TMEM_COLS - Tp) : 0u;
          const uint64_t a = ring_desc + (uint64_t)(((size_t)s * STAGE) >> 4);
          const uint64_t b = a + (uint64_t)(A_BYTES >> 4);
          const uint32_t acc0 = kb ? 1u : 0u;
          mma_stage(tmem + base, a, b, p.idesc, acc0);
          if (p.nmma == 2) mma_stage(tmem + base + (uint32_t)p.Nh, a, b + (uint64_t)((p.Nh * 128) >> 4), p.idesc, acc0);
          tc_commit(&empty[s]);
          if (kb == KB - 1) tc_commit(acc_full);
          ++issued;
        }
        __syncwarp();
      }
    }
    if (warp == MMA_WARP && lane == 0 && issued > 0) {
      // Every MMA this thread issued completes before TMEM is released.
      tc_commit(mma_done);
      volatile int dummy = 0;
      mbar_wait(mma_done, 0, &dummy, p.err, SITE_LMH_DRAIN, p.limit_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp;  // TMEM lane quarter: vocabulary rows 32q .. 32q+31 of the tile
    const int tid = threadIdx.x;  // 0..127
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int G = Tp / 32;
    const int n_ovl = 2 * Tp > TMEM_COLS ? (2 * Tp - TMEM_COLS) / 32 : 0;
    pdl_wait();  // drafts come from, and the outputs are read by, neighbouring kernels
    if (MODE == MODE_SAMPLED) {
      for (int c = tid; c < Tp; c += 128) {
        int d = -1;
        if (c < p.Mt) {
          const int b = c / (p.D + 1), j = c - b * (p.D + 1);
          if (j < p.D) d = p.draft[(size_t)b * p.D + j];
        }
        sdraft[c] = d;
      }
      named_barrier_sync(EPI_BAR_ID, 128);
    }
    for (int lt = 0; lt < my_tiles; ++lt) {
      const int t = (int)blockIdx.x + lt * (int)gridDim.x;
      const int v = t * BMV + 32 * q + lane;
      const bool valid = v < p.V;
      const bool ok = mbar_wait(acc_full, (uint32_t)lt & 1u, abort_flag, p.err, SITE_LMH_ACCFULL, p.limit_ns);
      if (named_barrier_or(EPI_BAR_ID, 128, ok ? 0u : 1u)) break;
      tc_fence_after();
      const uint32_t base = (lt & 1) ? (uint32_t)(TMEM_COLS - Tp) : 0u;
      const int start = ((lt & 1) == 0 && n_ovl) ? (TMEM_COLS - Tp) / 32 : 0;
      if (n_ovl == 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free);
      }
      for (int gi = 0; gi < G; ++gi) {
        int g = start + gi;
        if (g >= G) g -= G;
        const int c0 = 32 * g;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + base + (uint32_t)c0, r);
        tc_wait_ld();
        if (gi + 1 == n_ovl) {
          // The columns the next tile shares are in registers: release them.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_free);
        }
        if (MODE == MODE_LOGITS) {
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int c = c0 + i;
              if (c < p.Mt) p.logits[(size_t)c * p.ldl + v] = __float2bfloat16_rn(__uint_as_float(r[i]));
            }
          }
        } else {
          uint32_t key[32];
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const __nv_bfloat16 hb = __float2bfloat16_rn(__uint_as_float(r[i]));
            const uint32_t bits = (uint32_t)__bfloat16_as_ushort(hb);
            key[i] = valid ? ((ord16(bits) << 16) | (0xFFFFu - (uint32_t)(32 * q + lane))) : 0u;
            x[i] = __uint_as_float(bits << 16);
            if (MODE == MODE_SAMPLED && sdraft[c0 + i] == v) p.dl[c0 + i] = x[i];
          }
          const uint32_t kmax = transpose_reduce32(key, lane, MaxOp());
          float s = 0.f;
          if (MODE == MODE_SAMPLED) {
            float e[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t km = __shfl_sync(0xffffffffu, kmax, i);
              e[i] = valid ? exp2f((x[i] - key_value(km)) * p.k2) : 0.f;
            }
            s = transpose_reduce32(e, lane, AddOp());
          }
          part[q * Tp + c0 + lane] = make_uint2(kmax, __float_as_uint(s));
        }
      }
      if (MODE != MODE_LOGITS) {
        named_barrier_sync(EPI_BAR_ID, 128);
        for (int c = tid; c < p.Mt; c += 128) {
          uint2 a[4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) a[qq] = part[qq * Tp + c];
          uint32_t K = a[0].x;
#pragma unroll
          for (int qq = 1; qq < 4; ++qq) K = a[qq].x > K ? a[qq].x : K;
          float ssum = 0.f;
          if (MODE == MODE_SAMPLED) {
            const float m = key_value(K);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              if (a[qq].x) ssum += __uint_as_float(a[qq].y) * exp2f((key_value(a[qq].x) - m) * p.k2);
          }
          p.rec[(size_t)c * p.n_vt + t] = make_uint2(K, __float_as_uint(ssum));
        }
        named_barrier_sync(EPI_BAR_ID, 128);
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

// ------------------------------------------------------------ finalize

struct RowResult {
  int argmax;
  float p;      // softmax probability of the draft (T > 0)
  float m;      // the row's largest logit (T > 0)
  float s;      // the row's sum of exp((l - m) / T) (T > 0)
};

struct FinParams {
  uint2* rec;
  float* dl;
  int n_vt;
  int B, D;
  float k2;
  const int32_t* draft;
  const float* u;
  int32_t* n_acc;
  int32_t* next;
  RowResult* rows;   // [B*(D+1)]
  unsigned int* cnt; // [B], zero between calls
  // MODE_SAMPLE_NEXT: the lossless next token
  const float* u_next;
  const __nv_bfloat16* H;
  long long ldh;
  const uint8_t* wp;
  int K, KB, V;
};

constexpr int FIN_THREADS = 256;

// Exclusive prefix sum of one float per thread over the block, in thread
// order (a fixed order: the result is deterministic); returns the total.
QUASAR_DEVICE_INLINE float block_exclusive_scan(float x, float* s_warp, float& excl) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  float before = 0.f, total = 0.f;
  for (int k = 0; k < FIN_THREADS / 32; ++k) {
    if (k < w) before += s_warp[k];
    total += s_warp[k];
  }
  __syncthreads();
  excl = before + incl - x;
  return total;
}

// The lossless next token for T > 0 (the rule of quasar_verify_sample): a
// draw by inverse CDF on u_next from row n's softmax without the rejected
// draft (n < D) or from the bonus row (n = D).  The tile records give each
// vocabulary tile's weight; the tile holding u_next x total is found by a
// prefix sum in tile order, and its 128 logits are recomputed from the
// packed weight (fp32 sums, one rounding to BF16) for the walk inside it.
QUASAR_DEVICE_INLINE void draw_next(const FinParams& f, int b, int n, float* s_warp, float* s_f, int* s_i) {
  const int tid = threadIdx.x;
  const int R = f.D + 1;
  const int cr = b * R + n;
  const float m = __ldcg(&f.rows[cr].m);
  const int dr = n < f.D ? __ldcg(&f.draft[(size_t)b * f.D + n]) : -1;
  const float wd = dr >= 0 ? exp2f((__ldcg(&f.dl[cr]) - m) * f.k2) : 0.f;
  const uint2* rec = f.rec + (size_t)cr * f.n_vt;
  // Tile weights: thread tid owns the contiguous tiles [t0, t1).
  const int per = (f.n_vt + FIN_THREADS - 1) / FIN_THREADS;
  const int t0 = min(tid * per, f.n_vt), t1 = min(t0 + per, f.n_vt);
  float mine = 0.f;
  for (int t = t0; t < t1; ++t) {
    const uint2 r = __ldcg(&rec[t]);
    float wt = __uint_as_float(r.y) * exp2f((key_value(r.x) - m) * f.k2);
    if (dr >= 0 && t == dr / BMV) wt = fmaxf(wt - wd, 0.f);
    mine += wt;
  }
  float excl;
  const float total = block_exclusive_scan(mine, s_warp, excl);
  if (tid == 0) {
    s_i[0] = -1;
    s_i[1] = -1;
  }
  __syncthreads();
  if (!(total > 0.f)) {  // no weight left: the lowest index other than the draft
    if (tid == 0) f.next[b] = dr == 0 ? 1 : 0;
    return;
  }
  const float target = __ldcg(&f.u_next[b]) * total;
  {
    float run = excl;
    for (int t = t0; t < t1; ++t) {
      const uint2 r = __ldcg(&rec[t]);
      float wt = __uint_as_float(r.y) * exp2f((key_value(r.x) - m) * f.k2);
      if (dr >= 0 && t == dr / BMV) wt = fmaxf(wt - wd, 0.f);
      if (wt > 0.f) {
        if (run + wt > target) {
          atomicMin(reinterpret_cast<unsigned int*>(&s_i[0]), (unsigned int)t);  // -1 is the largest
          break;
        }
        atomicMax(&s_i[1], t);  // last tile with weight (rounding fallback)
      }
      run += wt;
    }
  }
  __syncthreads();
  const int ts = s_i[0] >= 0 ? s_i[0] : s_i[1];
  // cumulative weight before tile ts, recomputed in the same order by its owner
  if (tid == 0) s_f[0] = 0.f;
  __syncthreads();
  if (ts >= t0 && ts < t1) {
    float run = excl;
    for (int t = t0; t < ts; ++t) {
      const uint2 r = __ldcg(&rec[t]);
      float wt = __uint_as_float(r.y) * exp2f((key_value(r.x) - m) * f.k2);
      if (dr >= 0 && t == dr / BMV) wt = fmaxf(wt - wd, 0.f);
      run += wt;
    }
    s_f[0] = run;
  }
  // Recompute the tile's logits for token row cr: two threads per row, each
  // half of the K blocks of the packed weight.
  const int r = tid & (BMV - 1), kh = tid >> 7;
  const int kb0 = kh * ((f.KB + 1) / 2), kb1 = min(f.KB, kb0 + (f.KB + 1) / 2);
  const __nv_bfloat16* hrow = f.H + (size_t)cr * f.ldh;
  float acc = 0.f;
  for (int kb = kb0; kb < kb1; ++kb) {
    const uint8_t* wrow = f.wp + ((size_t)ts * f.KB + kb) * A_BYTES + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int k0 = kb * BKE + 8 * c;
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wrow + ((c ^ (r & 7)) << 4)));
      const __nv_bfloat16* wb = reinterpret_cast<const __nv_bfloat16*>(&wv);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (k0 + e < f.K) acc += __bfloat162float(wb[e]) * __bfloat162float(hrow[k0 + e]);
    }
  }
  s_f[8 + tid] = acc;
  __syncthreads();
  float e = 0.f;
  if (tid < BMV) {
    const int v = ts * BMV + tid;
    const float x = __bfloat162float(__float2bfloat16_rn(s_f[8 + tid] + s_f[8 + BMV + tid]));
    e = (v < f.V && v != dr) ? exp2f((x - m) * f.k2) : 0.f;
  }
  float ex;
  block_exclusive_scan(tid < BMV ? e : 0.f, s_warp, ex);
  const float tgt = target - s_f[0];
  if (tid == 0) {
    s_i[2] = -1;
    s_i[3] = -1;
  }
  __syncthreads();
  if (tid < BMV && e > 0.f) {
    if (ex + e > tgt) atomicMin(reinterpret_cast<unsigned int*>(&s_i[2]), (unsigned int)tid);
    atomicMax(&s_i[3], tid);
  }
  __syncthreads();
  if (tid == 0) {
    int v = s_i[2] >= 0 ? s_i[2] : s_i[3];
    if (v >= 0) {
      v += ts * BMV;
    } else {  // the recomputed tile has no weight left (rounding): the row's argmax, else the lowest non-draft index
      v = __ldcg(&f.rows[cr].argmax);
      if (v == dr) v = dr == 0 ? 1 : 0;
    }
    f.next[b] = v;
  }
}

template <int MODE>
__global__ void __launch_bounds__(FIN_THREADS) lm_head_finalize_kernel(const FinParams f) {
  constexpr bool SAMPLED = MODE == MODE_SAMPLED || MODE == MODE_SAMPLE_NEXT;
  constexpr bool KEEP = MODE == MODE_SAMPLE_NEXT;  // records stay until the draw
  __shared__ uint32_t s_ord[FIN_THREADS / 32];
  __shared__ int s_idx[FIN_THREADS / 32];
  __shared__ float s_sum[FIN_THREADS / 32];
  __shared__ float s_f[8 + FIN_THREADS];
  __shared__ int s_i[4];
  __shared__ int s_last, s_n;
  pdl_wait();
  const int c = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  uint2* rec = f.rec + (size_t)c * f.n_vt;

  // Pass 1: the largest logit and the lowest vocabulary index holding it.
  uint32_t bo = 0;
  int bi = INT_MAX;
  for (int t = tid; t < f.n_vt; t += FIN_THREADS) {
    const uint32_t k = __ldcg(&rec[t].x);
    if (!SAMPLED) rec[t] = make_uint2(0u, 0u);  // leave the workspace zero-filled
    const uint32_t o = k >> 16;
    const int idx = t * BMV + (int)(0xFFFFu - (k & 0xFFFFu));
    if (o > bo || (o == bo && idx < bi)) {
      bo = o;
      bi = idx;
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const uint32_t o2 = __shfl_xor_sync(0xffffffffu, bo, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, off);
    if (o2 > bo || (o2 == bo && i2 < bi)) {
      bo = o2;
      bi = i2;
    }
  }
  if (lane == 0) {
    s_ord[w] = bo;
    s_idx[w] = bi;
  }
  __syncthreads();
  bo = s_ord[0];
  bi = s_idx[0];
  for (int k = 1; k < FIN_THREADS / 32; ++k)
    if (s_ord[k] > bo || (s_ord[k] == bo && s_idx[k] < bi)) {
      bo = s_ord[k];
      bi = s_idx[k];
    }

  const int R = f.D + 1;
  const int b = c / R, j = c - b * R;
  float pj = 0.f, m = 0.f, tot = 0.f;
  if (SAMPLED) {
    // Pass 2: the row's sum of exp((l - max) / T), tile sums rescaled to the
    // row maximum, in a fixed order.
    m = key_value(bo << 16);
    float s = 0.f;
    for (int t = tid; t < f.n_vt; t += FIN_THREADS) {
      const uint2 r = __ldcg(&rec[t]);
      if (!KEEP) rec[t] = make_uint2(0u, 0u);
      s += __uint_as_float(r.y) * exp2f((key_value(r.x) - m) * f.k2);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    __syncthreads();  // s_ord / s_idx reads above are done before s_sum is written
    if (lane == 0) s_sum[w] = s;
    __syncthreads();
    for (int k = 0; k < FIN_THREADS / 32; ++k) tot += s_sum[k];
    if (j < f.D && tid == 0) {
      pj = exp2f((__ldcg(&f.dl[c]) - m) * f.k2) / tot;
      if (!KEEP) f.dl[c] = 0.f;
    }
  }

  if (tid == 0) {
    f.rows[c] = RowResult{bi, pj, m, tot};
    __threadfence();
    const unsigned int prev = atomicAdd(&f.cnt[b], 1u);
    s_last = (prev == (unsigned int)(R - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) {
    int n = f.D;
    for (int jj = 0; jj < f.D; ++jj) {
      const int am = __ldcg(&f.rows[b * R + jj].argmax);
      const float pr = __ldcg(&f.rows[b * R + jj].p);
      bool okj;
      if (SAMPLED)
        okj = __ldcg(&f.u[(size_t)b * f.D + jj]) < pr;
      else
        okj = __ldcg(&f.draft[(size_t)b * f.D + jj]) == am;
      if (!okj) {
        n = jj;
        break;
      }
    }
    f.n_acc[b] = n;
    if (!SAMPLED && f.next) f.next[b] = __ldcg(&f.rows[b * R + n].argmax);
    s_n = n;
  }
  __syncthreads();
  if (MODE == MODE_SAMPLE_NEXT) {
    draw_next(f, b, s_n, s_sum, s_f, s_i);
    __syncthreads();
    // the records and draft logits of this sequence's rows were kept for
    // the draw: zero them now
    for (size_t i = tid; i < (size_t)R * f.n_vt; i += FIN_THREADS) f.rec[(size_t)b * R * f.n_vt + i] = make_uint2(0u, 0u);
    for (int jj = tid; jj < R; jj += FIN_THREADS) f.dl[b * R + jj] = 0.f;
  }
  if (tid == 0) {
    for (int jj = 0; jj < R; ++jj) f.rows[b * R + jj] = RowResult{0, 0.f, 0.f, 0.f};
    f.cnt[b] = 0;
  }
}

// ------------------------------------------------------------ host side

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static int pad32(int m) { return (m + 31) & ~31; }

static int stages_for(int Tp) {
  int s = (int)((SMEM_LIMIT - smem_bytes(Tp, 0)) / stage_bytes(Tp));
  return s > MAX_STAGES ? MAX_STAGES : s;
}

size_t verify_workspace_size(int B, int D, int V) {
  if (B <= 0 || D < 0 || V <= 0) return 256;
  const size_t rows = (size_t)B * (D + 1);
  const size_t n_vt = (size_t)(V + BMV - 1) / BMV;
  return align256((size_t)B * 4) + align256(rows * sizeof(RowResult)) + align256(rows * 4) +
         align256(rows * n_vt * 8);
}

template <int MODE>
static cudaError_t launch_main(const CUtensorMap& th, const Params& p, int grid, cudaStream_t stream) {
  const uint32_t smem = smem_bytes(p.Tp, p.stages);
  static int configured[64] = {0};  // per device: the opt-in shared-memory size is set once
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(lm_head_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lm_head_kernel<MODE>, th, p);
}

template <int MODE>
static cudaError_t launch_fin(const FinParams& f, int rows, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(FIN_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lm_head_finalize_kernel<MODE>, f);
}

// Shared argument checks and the main kernel's parameters.
static quasar_status_t setup(const void* H, long long ldh, const void* Wp, int Mt, int V, int K, CUtensorMap* th,
                             Params* p, int* grid) {
  if (Mt < 0 || V <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (Mt > MAX_ROWS || K % 8 != 0 || ldh < K || ldh % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (!H || !Wp) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(H, 16) || !aligned(Wp, 16)) return QUASAR_ERR_UNSUPPORTED;
  Params& q = *p;
  q = Params{};
  q.Mt = Mt;
  q.Tp = pad32(Mt);
  q.nmma = q.Tp > 256 ? 2 : 1;
  q.Nh = q.Tp / q.nmma;  // multiple of 16, <= 256
  q.V = V;
  q.K = K;
  q.n_vt = (V + BMV - 1) / BMV;
  q.KB = (K + BKE - 1) / BKE;
  q.stages = stages_for(q.Tp);
  if (q.stages < 2) return QUASAR_ERR_UNSUPPORTED;
  q.wp = reinterpret_cast<const uint8_t*>(Wp);
  // kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B BF16
  // (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at 24.
  q.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(q.Nh >> 3) << 17) | ((uint32_t)(BMV >> 4) << 24);
  q.err = device_error_word();
  q.limit_ns = wait_limit_ns();
  if (!q.err) return QUASAR_ERR_CUDA;
  if (!encode_2d_bf16(th, H, K, Mt, ldh, BKE, q.Nh)) return QUASAR_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return QUASAR_ERR_CUDA;
  *grid = q.n_vt < sms ? q.n_vt : sms;
  return QUASAR_OK;
}

quasar_status_t run_logits(const void* H, int ldh, const void* Wp, int M, int V, int K, void* logits,
                           long long ldl, cudaStream_t stream) {
  if (M < 0 || V <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (ldl < V) return QUASAR_ERR_UNSUPPORTED;
  if (M == 0) return QUASAR_OK;
  if (!logits) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(logits, 2)) return QUASAR_ERR_UNSUPPORTED;
  CUtensorMap th;
  Params p;
  int grid = 0;
  quasar_status_t st = setup(H, ldh, Wp, M, V, K, &th, &p, &grid);
  if (st != QUASAR_OK) return st;
  p.logits = reinterpret_cast<__nv_bfloat16*>(logits);
  p.ldl = ldl;
  return cuda_status(launch_main<MODE_LOGITS>(th, p, grid, stream));
}

quasar_status_t run_verify(const void* H, int ldh, const void* Wp, int K, const int32_t* draft, int B, int D, int V,
                           float temperature, const float* u, const float* u_next, int32_t* n_acc, int32_t* next,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (B < 0 || D < 0 || V <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !(temperature < INFINITY)) return QUASAR_ERR_INVALID_ARG;
  const bool sampled = temperature > 0.f;
  const bool draw = u_next != nullptr;  // T > 0 with the lossless next token
  if (draw && (!sampled || !next)) return QUASAR_ERR_INVALID_ARG;
  if (B == 0) return QUASAR_OK;
  if ((long long)B * (D + 1) > MAX_ROWS) return QUASAR_ERR_UNSUPPORTED;
  if (!n_acc || (D > 0 && !draft) || (sampled && D > 0 && !u) || (sampled && !draw && next))
    return QUASAR_ERR_INVALID_ARG;
  if (!ws || ws_bytes < verify_workspace_size(B, D, V) || !aligned(ws, 256)) return QUASAR_ERR_WORKSPACE;
  const int Mt = B * (D + 1);
  CUtensorMap th;
  Params p;
  int grid = 0;
  quasar_status_t st = setup(H, ldh, Wp, Mt, V, K, &th, &p, &grid);
  if (st != QUASAR_OK) return st;

  uint8_t* w8 = reinterpret_cast<uint8_t*>(ws);
  unsigned int* cnt = reinterpret_cast<unsigned int*>(w8);
  w8 += align256((size_t)B * 4);
  RowResult* rows = reinterpret_cast<RowResult*>(w8);
  w8 += align256((size_t)Mt * sizeof(RowResult));
  float* dl = reinterpret_cast<float*>(w8);
  w8 += align256((size_t)Mt * 4);
  uint2* rec = reinterpret_cast<uint2*>(w8);

  p.rec = rec;
  p.dl = dl;
  p.draft = draft;
  p.D = D;
  p.k2 = sampled ? 1.4426950408889634f / temperature : 0.f;

  FinParams f;
  f.rec = rec;
  f.dl = dl;
  f.n_vt = p.n_vt;
  f.B = B;
  f.D = D;
  f.k2 = p.k2;
  f.draft = draft;
  f.u = u;
  f.n_acc = n_acc;
  f.next = next;
  f.rows = rows;
  f.cnt = cnt;
  f.u_next = u_next;
  f.H = reinterpret_cast<const __nv_bfloat16*>(H);
  f.ldh = ldh;
  f.wp = p.wp;
  f.K = K;
  f.KB = p.KB;
  f.V = V;

  cudaError_t e;
  if (sampled) {
    e = launch_main<MODE_SAMPLED>(th, p, grid, stream);
    if (e == cudaSuccess)
      e = draw ? launch_fin<MODE_SAMPLE_NEXT>(f, Mt, stream) : launch_fin<MODE_SAMPLED>(f, Mt, stream);
  } else {
    e = launch_main<MODE_GREEDY>(th, p, grid, stream);
    if (e == cudaSuccess) e = launch_fin<MODE_GREEDY>(f, Mt, stream);
  }
  return cuda_status(e);
}

// ------------------------------------------------------------ offline packing

size_t packed_bytes(int V, int K) {
  if (V <= 0 || K <= 0) return 0;
  return (size_t)((V + BMV - 1) / BMV) * (size_t)((K + BKE - 1) / BKE) * A_BYTES;
}

// One thread per 16-byte chunk of the packed weight: block (t, kb), row r,
// position pos holds the K values kb*64 + 8c .. +8 of vocabulary row
// t*128 + r with c = pos ^ (r % 8); chunks past V or K are zero.
__global__ void pack_kernel(const uint4* __restrict__ W, long long ldw16, int V, int K8, int KB, long long chunks,
                            uint4* __restrict__ out) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(i & 7);
    const int r = (int)((i >> 3) & (BMV - 1));
    const long long blk = i >> 10;  // 128 rows x 8 chunks per block
    const int kb = (int)(blk % KB);
    const long long t = blk / KB;
    const long long v = t * BMV + r;
    const int c8 = kb * 8 + (pos ^ (r & 7));  // 16-byte chunk index along K
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (v < V && c8 < K8) val = W[v * ldw16 + c8];
    out[i] = val;
  }
}

quasar_status_t run_pack(const void* W, int ldw, int V, int K, void* Wp, cudaStream_t stream) {
  if (V <= 0 || K <= 0) return QUASAR_ERR_INVALID_ARG;
  if (K % 8 != 0 || ldw < K || ldw % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (!W || !Wp) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(Wp, 16)) return QUASAR_ERR_UNSUPPORTED;
  const long long chunks = (long long)(packed_bytes(V, K) / 16);
  const int sms = sm_count();
  if (sms <= 0) return QUASAR_ERR_CUDA;
  pack_kernel<<<sms * 8, 256, 0, stream>>>(reinterpret_cast<const uint4*>(W), ldw / 8, V, K / 8,
                                          (K + BKE - 1) / BKE, chunks, reinterpret_cast<uint4*>(Wp));
  return cuda_status(cudaGetLastError());
}

}  // namespace lmhead
}  // namespace quasar

extern "C" {

size_t quasar_lm_head_packed_bytes(int V, int K) { return quasar::lmhead::packed_bytes(V, K); }

quasar_status_t quasar_pack_lm_head(const void* W_bf16, int ldw, int V, int K, void* Wp, quasar_stream_t stream) {
  return quasar::lmhead::run_pack(W_bf16, ldw, V, K, Wp, reinterpret_cast<cudaStream_t>(stream));
}

size_t quasar_lm_head_verify_workspace_size(int B, int D, int V) {
  return quasar::lmhead::verify_workspace_size(B, D, V);
}

quasar_status_t quasar_lm_head_logits(const void* H_bf16, int ldh, const void* Wp, int M, int V, int K,
                                      void* logits_bf16, long long ldl, quasar_stream_t stream) {
  return quasar::lmhead::run_logits(H_bf16, ldh, Wp, M, V, K, logits_bf16, ldl,
                                    reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_lm_head_verify(const void* H_bf16, int ldh, const void* Wp, int K, const int32_t* draft,
                                      int B, int D, int V, float temperature, const float* u, int32_t* n_acc,
                                      int32_t* next_token, void* workspace, size_t ws_bytes,
                                      quasar_stream_t stream) {
  return quasar::lmhead::run_verify(H_bf16, ldh, Wp, K, draft, B, D, V, temperature, u, nullptr, n_acc, next_token,
                                    workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_lm_head_verify_sample(const void* H_bf16, int ldh, const void* Wp, int K,
                                             const int32_t* draft, int B, int D, int V, float temperature,
                                             const float* u, const float* u_next, int32_t* n_acc,
                                             int32_t* next_token, void* workspace, size_t ws_bytes,
                                             quasar_stream_t stream) {
  if (!u_next || !next_token || !(temperature > 0.f)) return QUASAR_ERR_INVALID_ARG;
  return quasar::lmhead::run_verify(H_bf16, ldh, Wp, K, draft, B, D, V, temperature, u, u_next, n_acc, next_token,
                                    workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
