// A5: verification of drafted tokens -> accepted prefix length.
//
// Quasar summary zh §2 "方法论" / ko §2 "방법론": the dequantized logits stay
// in high precision and the drafts are checked with (lossless) rejection
// sampling; pt §4: greedy (T = 0) acceptance length.  Row j of sequence b
// scores draft j; row D is the bonus position.
//   T == 0: ok_j = draft[b][j] == argmax_v logits[b][j][v] (lowest index on ties)
//   T  > 0: ok_j = u[b][j] < softmax(logits[b][j] / T)[draft[b][j]]   (fp32)
//   n_acc[b] = first j with !ok_j, else D; next[b] = argmax of row n_acc[b].
//
// The step is an HBM scan of B*(D+1)*V BF16 logits.  Each row is cut into S
// chunks so that about 8 x 152 CTAs stream it with 128-bit non-allocating
// loads, four per thread in flight; a CTA reduces its chunk to (max, first argmax, running max, sum of
// exp) and stores that record.  The last CTA of a sequence (an atomic count;
// nobody waits) merges the records of its D+1 rows in chunk order, which
// makes every result deterministic, then zeroes those records and the counter.
#include <climits>

#include "quasar_common.cuh"

namespace quasar {
namespace verify {

constexpr int THREADS = 256;
constexpr int LOADS = 4;          // 16-byte loads per thread in flight
constexpr int TARGET_CTAS = 8 * 152;
constexpr int MIN_CHUNK = 4096;
constexpr int MERGE_BATCH = 4;    // chunk records of a row loaded at once by the merging lane

struct __align__(16) Partial {   // read back as one float4
  float best;  // max logit in the chunk
  int idx;     // lowest index holding it
  float m;     // running max of logit / T (T > 0)
  float s;     // sum of exp(logit/T - m) over the chunk (T > 0)
};

// Chunks per row the workspace provides for (device independent).
static int chunks_for(long long rows, int V) {
  long long s = (TARGET_CTAS + rows - 1) / rows;
  long long smax = (V + MIN_CHUNK - 1) / MIN_CHUNK;
  s = s < smax ? s : smax;
  return s < 1 ? 1 : (int)s;
}

// Chunk length (multiple of 8 elements) and the number of non-empty chunks
// for s0 requested chunks.
static void chunk_geometry_s(int V, int s0, int* ch, int* S) {
  int len = (V + s0 - 1) / s0;
  len = (len + 7) & ~7;
  *ch = len;
  *S = (V + len - 1) / len;
}

static void chunk_geometry(long long rows, int V, int* ch, int* S) { chunk_geometry_s(V, chunks_for(rows, V), ch, S); }

QUASAR_DEVICE_INLINE uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Count one finished chunk: release (this thread's record is visible before
// the count) and acquire (the CTA that takes the last count sees every
// record), one operation instead of a full fence and a relaxed atomic.
QUASAR_DEVICE_INLINE unsigned int count_acq_rel(unsigned int* p) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

QUASAR_DEVICE_INLINE void arg_merge(float& b, int& i, float b2, int i2) {
  if (b2 > b || (b2 == b && i2 < i)) {
    b = b2;
    i = i2;
  }
}

QUASAR_DEVICE_INLINE void lse_merge(float& m, float& s, float m2, float s2) {
  if (s2 == 0.f) return;
  if (s == 0.f) {
    m = m2;
    s = s2;
    return;
  }
  const float M = fmaxf(m, m2);
  s = s * expf(m - M) + s2 * expf(m2 - M);
  m = M;
}

// Lossless next token of sequence b (whole CTA): an inverse-CDF draw with
// uniform un from row j's weights w(v) = exp(logit(v) / T - M), M the row
// max, without the rejected draft token when j < D.  The chunk holding the
// target comes from the chunk records (mass s_c * exp(m_c - M)); that chunk
// is then scanned: every thread sums a contiguous sub-range, a block prefix
// sum places the sub-ranges, and the last thread whose prefix does not
// exceed the target walks its sub-range to the first running sum above it
// (or its last positive weight), so the result always has positive weight.
// A row with no weight left draws the lowest index other than the draft.
template <int NTH>
__device__ void resample(const uint16_t* __restrict__ logits, int ldl, const int32_t* __restrict__ draft, int D,
                         int V, int CH, int S, float invT, int b, int j, float un, const Partial* __restrict__ part,
                         int32_t* __restrict__ next_token) {
  __shared__ float s_M, s_t;
  __shared__ int s_c, s_pick;
  __shared__ float s_wsum[NTH / 32];
  const size_t row = (size_t)b * (D + 1) + j;
  const Partial* pr = part + row * S;
  const uint16_t* src = logits + row * ldl;
  const int dx = j < D ? draft[(size_t)b * D + j] : -1;
  const bool excl = dx >= 0 && dx < V;
  const int tid = threadIdx.x;
  auto mass = [&](int c, float M, float wd) {
    const float sc = __ldcg(&pr[c].s);
    float a = sc > 0.f ? sc * expf(__ldcg(&pr[c].m) - M) : 0.f;
    if (excl && c == dx / CH) a = fmaxf(a - wd, 0.f);
    return a;
  };
  if (tid == 0) {
    float M = -INFINITY;
    for (int c = 0; c < S; ++c)
      if (__ldcg(&pr[c].s) > 0.f) M = fmaxf(M, __ldcg(&pr[c].m));
    const float wd = excl ? expf(__uint_as_float((uint32_t)src[dx] << 16) * invT - M) : 0.f;
    float Z = 0.f;
    for (int c = 0; c < S; ++c) Z += mass(c, M, wd);
    const float target = un * Z;
    float A = 0.f;
    int cs = -1;
    for (int c = 0; c < S; ++c) {
      const float a = mass(c, M, wd);
      if (a > 0.f) cs = c;
      if (a > 0.f && A + a > target) break;
      A += a;
    }
    s_M = M;
    s_c = Z > 0.f ? cs : -1;
    s_t = target - A;
    s_pick = -1;
  }
  __syncthreads();
  if (s_c < 0) {   // no weight left
    if (tid == 0) next_token[b] = dx == 0 ? 1 : 0;
    return;
  }
  const float M = s_M, t = s_t;
  const int c0 = s_c * CH, c1 = min(V, c0 + CH);
  const int per = (c1 - c0 + NTH - 1) / NTH;
  const int v0 = min(c1, c0 + tid * per), v1 = min(c1, v0 + per);
  auto w = [&](int v) { return v == dx ? 0.f : expf(__uint_as_float((uint32_t)src[v] << 16) * invT - M); };
  float loc = 0.f;
  for (int v = v0; v < v1; ++v) loc += w(v);
  // Block exclusive prefix of the sub-range sums (fixed shape: deterministic).
  const int lane = tid & 31, wp = tid >> 5;
  float inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) s_wsum[wp] = inc;
  __syncthreads();
  float pre = inc - loc;
  for (int q = 0; q < wp; ++q) pre += s_wsum[q];
  if (loc > 0.f && pre <= t) atomicMax(&s_pick, tid);
  __syncthreads();
  // A chunk whose recorded mass was only rounding left over from the
  // removed draft holds no weight when rescanned: fall back as for an empty row.
  if (s_pick < 0 && tid == 0) next_token[b] = dx == 0 ? 1 : 0;
  if (tid == s_pick) {
    float run = pre;
    int got = -1, last = -1;
    for (int v = v0; v < v1; ++v) {
      const float x = w(v);
      if (x > 0.f) last = v;
      run += x;
      if (x > 0.f && run > t) {
        got = v;
        break;
      }
    }
    next_token[b] = got >= 0 ? got : last;
  }
}

template <bool SAMPLED>
__global__ void __launch_bounds__(THREADS)
verify_kernel(const uint16_t* __restrict__ logits, int ldl, const int32_t* __restrict__ draft, int D, int V,
              int CH, int S, float invT, const float* __restrict__ u, const float* __restrict__ u_next,
              int32_t* __restrict__ n_acc, int32_t* __restrict__ next_token, Partial* __restrict__ part,
              unsigned int* __restrict__ cnt) {
  // Launched with programmatic dependent launch: the CTAs start while the
  // previous kernel drains and wait here for its writes (the logits).
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.y;
  const int c = blockIdx.x;
  const int b = row / (D + 1);
  const uint16_t* src = logits + (size_t)row * ldl;
  const int start = c * CH;
  const int end = min(V, start + CH);
  const int vend = start + ((end - start) / 8) * 8;

  float best = -INFINITY;
  int idx = INT_MAX;
  float m = -INFINITY, s = 0.f;
  auto take = [&](float f, int k) {
    if (f > best) {
      best = f;
      idx = k;
    }
    if (SAMPLED) {
      const float z = f * invT;
      if (z > m) {
        s = s * expf(m - z) + 1.f;
        m = z;
      } else {
        s += expf(z - m);
      }
    }
  };
  auto take8 = [&](const uint4& raw, int v) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      take(__uint_as_float(w[i] << 16), v + 2 * i);
      take(__uint_as_float(w[i] & 0xFFFF0000u), v + 2 * i + 1);
    }
  };
  // LOADS loads of each thread in flight before any is used (one load per
  // step left too few bytes in flight per SM to cover HBM latency); each
  // thread still takes its elements in increasing index order.
  int v = start + threadIdx.x * 8;
  for (; v + (LOADS - 1) * THREADS * 8 < vend; v += LOADS * THREADS * 8) {
    uint4 raw[LOADS];
#pragma unroll
    for (int i = 0; i < LOADS; ++i) raw[i] = ld_stream(src + v + i * THREADS * 8);
#pragma unroll
    for (int i = 0; i < LOADS; ++i) take8(raw[i], v + i * THREADS * 8);
  }
  for (; v < vend; v += THREADS * 8) take8(ld_stream(src + v), v);
  for (int v = vend + threadIdx.x; v < end; v += THREADS) take(__uint_as_float((uint32_t)src[v] << 16), v);

  // Block reduction (fixed shape, so deterministic).
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    arg_merge(best, idx, b2, i2);
    if (SAMPLED) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
  }
  __shared__ Partial red[THREADS / 32];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = Partial{best, idx, m, s};
  __syncthreads();
  if (threadIdx.x == 0) {
    Partial r = red[0];
    for (int w = 1; w < THREADS / 32; ++w) {
      arg_merge(r.best, r.idx, red[w].best, red[w].idx);
      if (SAMPLED) lse_merge(r.m, r.s, red[w].m, red[w].s);
    }
    part[(size_t)row * S + c] = r;
    const unsigned int total = (unsigned int)(D + 1) * (unsigned int)S;
    const unsigned int old = count_acq_rel(&cnt[b]);
    is_last = (old + 1 == total) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;

  // Last CTA of sequence b: merge each row's chunk records in chunk order.
  // Thread 0's acquire-release count made every record of the sequence
  // visible to it, and the barrier above orders the loads below after it.
  // Each lane loads its row's draft token and every record of the row
  // before using any (one round trip, not one per record).
  __shared__ int s_fail;
  if (warp == 0) {
    int first_fail = D;
    int ri_row = INT_MAX;   // argmax of row `lane` (D < 32: one row per lane)
    for (int j = lane; j <= D; j += 32) {
      const Partial* pr = part + ((size_t)b * (D + 1) + j) * S;
      const int d = j < D ? draft[(size_t)b * D + j] : -1;
      float rb = -INFINITY, rm = -INFINITY, rs = 0.f;
      int ri = INT_MAX;
      for (int c0 = 0; c0 < S; c0 += MERGE_BATCH) {
        float4 rec[MERGE_BATCH];
#pragma unroll
        for (int k = 0; k < MERGE_BATCH; ++k)
          if (c0 + k < S) rec[k] = __ldcg(reinterpret_cast<const float4*>(pr + c0 + k));
#pragma unroll
        for (int k = 0; k < MERGE_BATCH; ++k) {
          if (c0 + k >= S) break;
          arg_merge(rb, ri, rec[k].x, __float_as_int(rec[k].y));
          if (SAMPLED) lse_merge(rm, rs, rec[k].z, rec[k].w);
        }
      }
      ri_row = ri;
      if (j < D) {
        bool ok;
        if (d < 0 || d >= V) {
          ok = false;  // out-of-vocabulary draft: rejected, never dereferenced
        } else if (SAMPLED) {
          const float ld = __uint_as_float((uint32_t)logits[((size_t)b * (D + 1) + j) * ldl + d] << 16);
          const float pj = __fdiv_rn(expf(ld * invT - rm), rs);
          ok = u[(size_t)b * D + j] < pj;
        } else {
          ok = (d == ri);
        }
        if (!ok) first_fail = min(first_fail, j);
      }
    }
  #pragma unroll
    for (int o = 16; o > 0; o >>= 1) first_fail = min(first_fail, __shfl_xor_sync(0xffffffffu, first_fail, o));
    const int ri_fail = __shfl_sync(0xffffffffu, ri_row, first_fail & 31);
    if (lane == 0) {
      n_acc[b] = first_fail;
      s_fail = first_fail;
      if (!SAMPLED && next_token && D < 32) {
        next_token[b] = ri_fail;   // lane first_fail merged that row above
      } else if (!SAMPLED && next_token) {
        const Partial* pr = part + ((size_t)b * (D + 1) + first_fail) * S;
        float rb = -INFINITY;
        int ri = INT_MAX;
        for (int cc = 0; cc < S; ++cc) arg_merge(rb, ri, __ldcg(&pr[cc].best), __ldcg(&pr[cc].idx));
        next_token[b] = ri;
      }
    }
  }
  if (SAMPLED && u_next) {
    __syncthreads();
    resample<THREADS>(logits, ldl, draft, D, V, CH, S, invT, b, s_fail, u_next[b], part, next_token);
  }
  // Leave the workspace zero-filled for the next call (its records and counter).
  __syncthreads();
  if (warp != 0) return;
  for (int j = lane; j <= D; j += 32) {
    Partial* pr = part + ((size_t)b * (D + 1) + j) * S;
    for (int cc = 0; cc < S; ++cc) __stcg(reinterpret_cast<float4*>(&pr[cc]), make_float4(0.f, 0.f, 0.f, 0.f));
  }
  if (lane == 0) atomicExch(&cnt[b], 0u);
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t workspace_size(int B, int D, int V) {
  if (B <= 0 || D < 0 || V <= 0) return 0;
  const long long rows = (long long)B * (D + 1);
  int ch, S;
  chunk_geometry(rows, V, &ch, &S);
  return align256((size_t)B * 4) + (size_t)rows * S * sizeof(Partial);
}

static quasar_status_t run(const void* logits_bf16, int ldl, const int32_t* draft, int B, int D, int V,
                           float temperature, const float* u, const float* u_next, int32_t* n_acc,
                           int32_t* next_token, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (B < 0 || D < 0 || V <= 0) return QUASAR_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || temperature == INFINITY) return QUASAR_ERR_INVALID_ARG;
  const bool sampled = temperature > 0.f;
  if (ldl < V || ldl % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (B == 0) return QUASAR_OK;  // no sequences: nothing is read or written
  if (!logits_bf16 || !n_acc || (D > 0 && !draft) || (sampled && D > 0 && !u)) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(logits_bf16, 16)) return QUASAR_ERR_UNSUPPORTED;
  if ((long long)B * (D + 1) > 65535) return QUASAR_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < workspace_size(B, D, V) || !aligned(workspace, 256)) return QUASAR_ERR_WORKSPACE;
  const long long rows = (long long)B * (D + 1);
  // As many chunks per row as fill one wave of resident CTAs (a second,
  // mostly empty wave would leave HBM idle), within the workspace's records.
  int ch, S;
  chunk_geometry(rows, V, &ch, &S);
  {
    int per_sm = 0;
    const cudaError_t e = sampled ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<true>, THREADS, 0)
                                  : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<false>, THREADS, 0);
    const long long resident = (long long)per_sm * sm_count();
    if (e == cudaSuccess && resident > 0) {
      const long long want = resident / rows;
      const int s0 = (int)(want < 1 ? 1 : (want < S ? want : S));
      chunk_geometry_s(V, s0, &ch, &S);
    } else {
      cudaGetLastError();
    }
  }
  unsigned int* cnt = reinterpret_cast<unsigned int*>(workspace);
  Partial* part = reinterpret_cast<Partial*>(reinterpret_cast<uint8_t*>(workspace) + align256((size_t)B * 4));
  const dim3 grid(S, (unsigned)rows);
  const float invT = sampled ? 1.0f / temperature : 0.f;
  const uint16_t* lg = reinterpret_cast<const uint16_t*>(logits_bf16);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      sampled ? cudaLaunchKernelEx(&cfg, verify_kernel<true>, lg, ldl, draft, D, V, ch, S, invT, u, u_next, n_acc,
                                   next_token, part, cnt)
              : cudaLaunchKernelEx(&cfg, verify_kernel<false>, lg, ldl, draft, D, V, ch, S, invT, u,
                                   static_cast<const float*>(nullptr), n_acc, next_token, part, cnt);
  return cuda_status(e);
}

}  // namespace verify
}  // namespace quasar

extern "C" {

size_t quasar_verify_accept_workspace_size(int B, int D, int V) { return quasar::verify::workspace_size(B, D, V); }

quasar_status_t quasar_verify_accept(const void* logits_bf16, int ldl, const int32_t* draft, int B, int D, int V,
                                     float temperature, const float* u, int32_t* n_acc, int32_t* next_token,
                                     void* workspace, size_t ws_bytes, quasar_stream_t stream) {
  if (temperature > 0.f && next_token) return QUASAR_ERR_INVALID_ARG;
  return quasar::verify::run(logits_bf16, ldl, draft, B, D, V, temperature, u, nullptr, n_acc, next_token, workspace,
                             ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

quasar_status_t quasar_verify_sample(const void* logits_bf16, int ldl, const int32_t* draft, int B, int D, int V,
                                     float temperature, const float* u, const float* u_next, int32_t* n_acc,
                                     int32_t* next_token, void* workspace, size_t ws_bytes, quasar_stream_t stream) {
  if (!(temperature > 0.f) || temperature == INFINITY) return QUASAR_ERR_INVALID_ARG;
  if (B > 0 && (!u_next || !next_token)) return QUASAR_ERR_INVALID_ARG;
  return quasar::verify::run(logits_bf16, ldl, draft, B, D, V, temperature, u, u_next, n_acc, next_token, workspace,
                             ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
