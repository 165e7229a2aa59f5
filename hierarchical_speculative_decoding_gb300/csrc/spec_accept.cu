// a8 -- lossless speculative accept / resample of one verification level.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "Dual Rejection
// Sampling: Mathematical Losslessness": drafted token x is kept when
// min(1, p(x)/q(x)) >= u; at the first rejection the verifier resamples from
// max(0, p - q) normalised; the two levels (tiny drafter -> retrieval drafter,
// retrieval drafter -> target) compose to the target distribution.
//
// Design: latency-bound, one CTA per sequence.  The CTA computes the softmax
// normaliser (max, sum of exponentials) of every row it may need, runs the
// sequential ratio tests on one thread in fp64, then draws the next token
// with an index-order inverse CDF: each thread owns a contiguous slice of the
// vocabulary, slice sums are scanned across the block in fp64, and the one
// thread whose slice holds the crossing walks it.
#include "tf_common.cuh"

namespace tf {
namespace {

constexpr int kMaxThreads = 1024;

// Softmax normaliser of a row in the log2 domain: x_t = logit_t * log2(e) / temperature.
struct RowNorm {
  float m;   // max_t x_t
  double z;  // sum_t 2^(x_t - m)
};

__device__ __forceinline__ void combine(float& m, float& z, float m2, float z2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  z = z * merge_scale(m, mn) + z2 * merge_scale(m2, mn);
  m = mn;
}

// Block-wide softmax normaliser of one row.  scratch: >= 2 * 32 floats.
__device__ RowNorm row_norm(const float* __restrict__ row, int V, float inv_t, float* s_m, double* s_z) {
  float m = -INFINITY, z = 0.0f;
  for (int t = threadIdx.x; t < V; t += blockDim.x) {
    const float x = row[t] * inv_t;
    if (x > m) {
      z = z * merge_scale(m, x) + 1.0f;
      m = x;
    } else {
      z += exp2f(x - m);
    }
  }
  // Warp combine in fp32 (few terms), block combine in fp64.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    combine(m, z, m2, z2);
  }
  const int warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    s_m[warp] = m;
    s_z[warp] = (double)z;
  }
  __syncthreads();
  RowNorm r;
  float mm = -INFINITY;
  for (int w = 0; w < nw; ++w) mm = fmaxf(mm, s_m[w]);
  double zz = 0.0;
  for (int w = 0; w < nw; ++w)
    if (s_m[w] != -INFINITY) zz += s_z[w] * exp2((double)s_m[w] - (double)mm);
  r.m = mm;
  r.z = zz;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kMaxThreads) spec_accept_kernel(
    const float* __restrict__ tgt, const float* __restrict__ drf, const int32_t* __restrict__ tokens,
    const float* __restrict__ u_acc, const float* __restrict__ u_res, int gamma, int V, float inv_t,
    double inv_t_d,
    int32_t* __restrict__ n_acc, int32_t* __restrict__ next_token, int32_t* __restrict__ out_tokens) {
  __shared__ float s_m[32];
  __shared__ double s_z[32];
  __shared__ double s_scan[32];
  __shared__ int s_g, s_nacc, s_next, s_found, s_last;
  const int b = blockIdx.x;
  const float* P = tgt + (size_t)b * (gamma + 1) * V;
  const float* Q = drf + (size_t)b * gamma * V;
  const int32_t* x = tokens + (size_t)b * gamma;

  if (threadIdx.x == 0) {
    int g = gamma;
    for (int i = 0; i < gamma; ++i)
      if (x[i] < 0 || x[i] >= V) { g = i; break; }
    s_g = g;
  }
  __syncthreads();
  const int g = s_g;

  // ---- sequential ratio tests (normalisers computed block-wide per row)
  int nacc = g;
  for (int i = 0; i < g; ++i) {
    const RowNorm np = row_norm(P + (size_t)i * V, V, inv_t, s_m, s_z);
    const RowNorm nq = row_norm(Q + (size_t)i * V, V, inv_t, s_m, s_z);
    if (threadIdx.x == 0) {
      const int xi = x[i];
      // The drafted token's own terms in fp64 from the raw logits.
      const double lp = (double)P[(size_t)i * V + xi] * inv_t_d - (double)np.m;
      const double lq = (double)Q[(size_t)i * V + xi] * inv_t_d - (double)nq.m;
      const double qx = exp2(lq) / nq.z;
      const double ratio = exp2(lp - lq) * (nq.z / np.z);
      const bool accept = (qx == 0.0) || ((double)u_acc[(size_t)b * gamma + i] <= ratio);
      s_nacc = accept ? -1 : i;
    }
    __syncthreads();
    if (s_nacc >= 0) { nacc = s_nacc; break; }
  }

  // ---- the sampling row: residual at the first rejection, else the bonus row
  const bool rejected = nacc < g;
  const int j = nacc;
  const RowNorm np = row_norm(P + (size_t)j * V, V, inv_t, s_m, s_z);
  RowNorm nq = np;
  if (rejected) nq = row_norm(Q + (size_t)j * V, V, inv_t, s_m, s_z);
  const float* pr = P + (size_t)j * V;
  const float* qr = Q + (size_t)j * V;
  const float inv_zp = (float)(1.0 / np.z), inv_zq = (float)(1.0 / nq.z);

  const int seg = (V + blockDim.x - 1) / blockDim.x;
  const int t0 = min(V, (int)threadIdx.x * seg), t1 = min(V, t0 + seg);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  const double u = (double)u_res[b];

  for (int attempt = 0; attempt < 2; ++attempt) {
    // attempt 0: residual (if rejected) or p_g; attempt 1: p_j when the residual is all zero
    const bool use_resid = rejected && attempt == 0;
    float run = 0.0f;
    for (int t = t0; t < t1; ++t) {
      const float pt = exp2f(pr[t] * inv_t - np.m) * inv_zp;
      float w = pt;
      if (use_resid) w = fmaxf(pt - exp2f(qr[t] * inv_t - nq.m) * inv_zq, 0.0f);
      run += w;
    }
    // fp64 exclusive scan of the slice sums
    double incl = (double)run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    double wpre = 0.0, total = 0.0;
    for (int w = 0; w < nw; ++w) {
      const double v = s_scan[w];
      if (w < warp) wpre += v;
      total += v;
    }
    const double excl = wpre + incl - (double)run;
    if (threadIdx.x == 0) {
      s_found = 0x7fffffff;
      s_last = -1;
    }
    __syncthreads();
    if (total > 0.0) {
      const double target = u * total;
      if (excl <= target && excl + (double)run > target) {
        float r2 = 0.0f;
        for (int t = t0; t < t1; ++t) {
          const float pt = exp2f(pr[t] * inv_t - np.m) * inv_zp;
          float w = pt;
          if (use_resid) w = fmaxf(pt - exp2f(qr[t] * inv_t - nq.m) * inv_zq, 0.0f);
          r2 += w;
          if (excl + (double)r2 > target) {
            atomicMin(&s_found, t);
            break;
          }
        }
      }
      __syncthreads();
      if (s_found == 0x7fffffff) {
        // Rounding left no crossing: take the last index with positive weight.
        int last = -1;
        for (int t = t0; t < t1; ++t) {
          const float pt = exp2f(pr[t] * inv_t - np.m) * inv_zp;
          float w = pt;
          if (use_resid) w = fmaxf(pt - exp2f(qr[t] * inv_t - nq.m) * inv_zq, 0.0f);
          if (w > 0.0f) last = t;
        }
        if (last >= 0) atomicMax(&s_last, last);
        __syncthreads();
        if (threadIdx.x == 0) s_found = s_last < 0 ? 0 : s_last;
      }
      __syncthreads();
      if (threadIdx.x == 0) s_next = s_found;
      __syncthreads();
      break;
    }
    __syncthreads();
    if (!use_resid) {
      if (threadIdx.x == 0) s_next = 0;
      __syncthreads();
      break;
    }
  }

  if (threadIdx.x == 0) {
    n_acc[b] = nacc;
    next_token[b] = s_next;
  }
  if (out_tokens) {
    for (int c = threadIdx.x; c <= gamma; c += blockDim.x) {
      int v = -1;
      if (c < nacc) v = x[c];
      else if (c == nacc) v = s_next;
      out_tokens[(size_t)b * (gamma + 1) + c] = v;
    }
  }
}

}  // namespace
}  // namespace tf

extern "C" tf_status tf_spec_accept(const float* tgt_logits, const float* drf_logits, const int32_t* drf_tokens,
                                    const float* u_acc, const float* u_res, int B, int gamma, int V,
                                    float temperature, int32_t* n_acc, int32_t* next_token, int32_t* out_tokens,
                                    tf_stream_t stream) {
  using namespace tf;
  if (!tgt_logits || !u_res || !n_acc || !next_token) return TF_ERR_INVALID_ARG;
  if (gamma > 0 && (!drf_logits || !drf_tokens || !u_acc)) return TF_ERR_INVALID_ARG;
  if (B < 0 || gamma < 0 || V < 1 || !(temperature > 0.0f)) return TF_ERR_INVALID_ARG;
  if (B == 0) return TF_OK;
  int threads = ((V / 8 + 31) / 32) * 32;
  if (threads < 32) threads = 32;
  if (threads > kMaxThreads) threads = kMaxThreads;
  const double inv_t_d = 1.4426950408889634 / (double)temperature;  // log2(e) / temperature
  spec_accept_kernel<<<B, threads, 0, stream>>>(tgt_logits, drf_logits, drf_tokens, u_acc, u_res, gamma, V,
                                                (float)inv_t_d, inv_t_d, n_acc, next_token, out_tokens);
  return launch_status();
}
