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
// loads; a CTA reduces its chunk to (max, first argmax, running max, sum of
// exp) and stores that record.  The last CTA of a sequence (an atomic count;
// nobody waits) merges the records of its D+1 rows in chunk order, which
// makes every result deterministic, then zeroes those records and the counter.
#include <climits>

#include "quasar_common.cuh"

namespace quasar {
namespace verify {

constexpr int THREADS = 256;
constexpr int TARGET_CTAS = 8 * 152;
constexpr int MIN_CHUNK = 4096;

struct Partial {
  float best;  // max logit in the chunk
  int idx;     // lowest index holding it
  float m;     // running max of logit / T (T > 0)
  float s;     // sum of exp(logit/T - m) over the chunk (T > 0)
};

static int chunks_for(long long rows, int V) {
  long long s = (TARGET_CTAS + rows - 1) / rows;
  long long smax = (V + MIN_CHUNK - 1) / MIN_CHUNK;
  s = s < smax ? s : smax;
  return s < 1 ? 1 : (int)s;
}

// Chunk length (multiple of 8 elements) and the number of non-empty chunks.
static void chunk_geometry(long long rows, int V, int* ch, int* S) {
  const int s0 = chunks_for(rows, V);
  int len = (V + s0 - 1) / s0;
  len = (len + 7) & ~7;
  *ch = len;
  *S = (V + len - 1) / len;
}

QUASAR_DEVICE_INLINE uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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

template <bool SAMPLED>
__global__ void __launch_bounds__(THREADS)
verify_kernel(const uint16_t* __restrict__ logits, int ldl, const int32_t* __restrict__ draft, int D, int V,
              int CH, int S, float invT, const float* __restrict__ u, int32_t* __restrict__ n_acc,
              int32_t* __restrict__ next_token, Partial* __restrict__ part, unsigned int* __restrict__ cnt) {
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
  for (int v = start + threadIdx.x * 8; v < vend; v += THREADS * 8) {
    const uint4 raw = ld_stream(src + v);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      take(__uint_as_float(w[i] << 16), v + 2 * i);
      take(__uint_as_float(w[i] & 0xFFFF0000u), v + 2 * i + 1);
    }
  }
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
    __threadfence();
    const unsigned int total = (unsigned int)(D + 1) * (unsigned int)S;
    const unsigned int old = atomicAdd(&cnt[b], 1u);
    is_last = (old + 1 == total) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last || warp != 0) return;

  // Last CTA of sequence b: merge each row's chunk records in chunk order.
  __threadfence();
  int first_fail = D;
  for (int j = lane; j <= D; j += 32) {
    const Partial* pr = part + ((size_t)b * (D + 1) + j) * S;
    float rb = -INFINITY, rm = -INFINITY, rs = 0.f;
    int ri = INT_MAX;
    for (int cc = 0; cc < S; ++cc) {
      const float pb = __ldcg(&pr[cc].best);
      const int pi = __ldcg(&pr[cc].idx);
      arg_merge(rb, ri, pb, pi);
      if (SAMPLED) lse_merge(rm, rs, __ldcg(&pr[cc].m), __ldcg(&pr[cc].s));
    }
    if (j < D) {
      const int d = draft[(size_t)b * D + j];
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
  if (lane == 0) {
    n_acc[b] = first_fail;
    if (!SAMPLED && next_token) {
      const Partial* pr = part + ((size_t)b * (D + 1) + first_fail) * S;
      float rb = -INFINITY;
      int ri = INT_MAX;
      for (int cc = 0; cc < S; ++cc) arg_merge(rb, ri, __ldcg(&pr[cc].best), __ldcg(&pr[cc].idx));
      next_token[b] = ri;
    }
  }
  // Leave the workspace zero-filled for the next call (its records and counter).
  __syncwarp();
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

}  // namespace verify
}  // namespace quasar

extern "C" {

size_t quasar_verify_accept_workspace_size(int B, int D, int V) { return quasar::verify::workspace_size(B, D, V); }

quasar_status_t quasar_verify_accept(const void* logits_bf16, int ldl, const int32_t* draft, int B, int D, int V,
                                     float temperature, const float* u, int32_t* n_acc, int32_t* next_token,
                                     void* workspace, size_t ws_bytes, quasar_stream_t stream_) {
  using namespace quasar;
  using namespace quasar::verify;
  if (B < 0 || D < 0 || V <= 0) return QUASAR_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || temperature == INFINITY) return QUASAR_ERR_INVALID_ARG;
  const bool sampled = temperature > 0.f;
  if (sampled && next_token) return QUASAR_ERR_INVALID_ARG;
  if (ldl < V || ldl % 8 != 0) return QUASAR_ERR_UNSUPPORTED;
  if (B == 0) return QUASAR_OK;  // no sequences: nothing is read or written
  if (!logits_bf16 || !n_acc || (D > 0 && !draft) || (sampled && D > 0 && !u)) return QUASAR_ERR_INVALID_ARG;
  if (!aligned(logits_bf16, 16)) return QUASAR_ERR_UNSUPPORTED;
  if ((long long)B * (D + 1) > 65535) return QUASAR_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < workspace_size(B, D, V) || !aligned(workspace, 256)) return QUASAR_ERR_WORKSPACE;
  const long long rows = (long long)B * (D + 1);
  int ch, S;
  chunk_geometry(rows, V, &ch, &S);
  unsigned int* cnt = reinterpret_cast<unsigned int*>(workspace);
  Partial* part = reinterpret_cast<Partial*>(reinterpret_cast<uint8_t*>(workspace) + align256((size_t)B * 4));
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const dim3 grid(S, (unsigned)rows);
  const float invT = sampled ? 1.0f / temperature : 0.f;
  const uint16_t* lg = reinterpret_cast<const uint16_t*>(logits_bf16);
  if (sampled)
    verify_kernel<true><<<grid, THREADS, 0, stream>>>(lg, ldl, draft, D, V, ch, S, invT, u, n_acc, nullptr, part,
                                                      cnt);
  else
    verify_kernel<false><<<grid, THREADS, 0, stream>>>(lg, ldl, draft, D, V, ch, S, invT, u, n_acc, next_token,
                                                       part, cnt);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
