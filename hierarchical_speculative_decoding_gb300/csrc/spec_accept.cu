// a8 -- lossless speculative accept / resample of one verification level.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "Dual Rejection
// Sampling: Mathematical Losslessness": drafted token x is kept when
// min(1, p(x)/q(x)) >= u; at the first rejection the verifier resamples from
// max(0, p - q) normalised; the two levels (tiny drafter -> retrieval drafter,
// retrieval drafter -> target) compose to the target distribution.
//
// Design: latency-bound, two short kernels chained with programmatic dependent
// launch.  (1) Every logit row that may be needed (gamma + 1 verifier rows and
// gamma drafter rows per sequence) gets its softmax normaliser -- max and sum of
// exponentials in the log2 domain -- from its own group of threads (a warp for
// small vocabularies, 512 threads otherwise), with all loads of a thread issued
// together.  (2) One group per sequence runs the ratio tests on one thread in
// fp64 from those normalisers and the drafted tokens' own logits, then draws the
// next token with an index-order inverse CDF: each thread owns a contiguous
// slice of the vocabulary, the slice sums are scanned across the group in fp64,
// and the thread whose slice holds the crossing walks it again.
#include "tf_common.cuh"

namespace tf {
namespace {

constexpr int kBlockRow = 512;   // threads per row normaliser for large vocabularies
constexpr int kBlockSeq = 1024;  // threads per sequence for large vocabularies
constexpr int kSmallV = 1024;    // up to this vocabulary a warp handles a row / a sequence
constexpr int kBatch = 8;        // loads in flight per thread
constexpr size_t kMaxStageBytes = 200 * 1024;  // staged sampling row (vocabularies up to ~48K)

struct NormWs {
  float* m;   // [B, R] max of x = logit * log2(e) / temperature
  double* z;  // [B, R] sum of 2^(x - m)
};

__device__ __forceinline__ void combine(float& m, float& z, float m2, float z2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  z = z * merge_scale(m, mn) + z2 * merge_scale(m2, mn);
  m = mn;
}

// hi + lo += bh + bl for unevaluated fp32 pairs (|lo| <= ulp(hi) / 2): TwoSum of
// the high parts, the low parts added to its error, renormalised.
__device__ __forceinline__ void pair_add(float& hi, float& lo, float bh, float bl) {
  const float s = hi + bh;
  const float bb = s - hi;
  float e = (hi - (s - bb)) + (bh - bb);
  e += lo + bl;
  hi = s + e;
  lo = e - (hi - s);
}

// Per-thread (max, sum) over elements t = start, start + stride, ... < V, NB
// loads in flight at a time.
template <int NB>
__device__ __forceinline__ void thread_norm(const float* __restrict__ row, int V, int start, int stride, float inv_t,
                                            float& m, float& z) {
  m = -INFINITY;
  z = 0.0f;
  for (int t0 = start; t0 < V; t0 += stride * NB) {
    float x[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int t = t0 + k * stride;
      x[k] = t < V ? __ldg(row + t) * inv_t : -INFINITY;
    }
    float bm = x[0];
#pragma unroll
    for (int k = 1; k < NB; ++k) bm = fmaxf(bm, x[k]);
    if (bm == -INFINITY) continue;
    float bz = 0.0f;
#pragma unroll
    for (int k = 0; k < NB; ++k) bz += exp2f(x[k] - bm);
    combine(m, z, bm, bz);
  }
}

// (1) Normaliser of every row.  Rows are numbered [b][r] with r < gamma+1 the
// verifier rows and r >= gamma+1 the drafter rows.  WARP: one warp per row.
template <bool WARP>
__global__ void __launch_bounds__(WARP ? 256 : kBlockRow) row_norm_kernel(const float* __restrict__ tgt,
                                                                          const float* __restrict__ drf, int B,
                                                                          int gamma, int V, float inv_t, NormWs ws) {
  pdl_wait();
  const int R = 2 * gamma + 1;
  long long row;
  int start, stride;
  if (WARP) {
    row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    start = threadIdx.x & 31;
    stride = 32;
  } else {
    row = blockIdx.x;
    start = threadIdx.x;
    stride = blockDim.x;
  }
  if (row >= (long long)B * R) return;  // a whole warp (or block) leaves together
  const int b = (int)(row / R), r = (int)(row % R);
  const float* src = r <= gamma ? tgt + ((size_t)b * (gamma + 1) + r) * V
                                : drf + ((size_t)b * gamma + (r - gamma - 1)) * V;
  float m, z;
  if (WARP)
    thread_norm<kBatch>(src, V, start, stride, inv_t, m, z);
  else
    thread_norm<4 * kBatch>(src, V, start, stride, inv_t, m, z);  // a 32000-entry row in two rounds
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    combine(m, z, m2, z2);
  }
  if (WARP) {
    if ((threadIdx.x & 31) == 0) {
      ws.m[row] = m;
      ws.z[row] = (double)z;
    }
    return;
  }
  __shared__ float s_m[32];
  __shared__ double s_z[32];
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_m[warp] = m;
    s_z[warp] = (double)z;
  }
  __syncthreads();
  if (warp == 0) {
    // the warps' states combined by one warp: max, then sum z_w 2^(m_w - max)
    const int lane = threadIdx.x & 31;
    const float mw = lane < nw ? s_m[lane] : -INFINITY;
    float mm = mw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    double zz = (mw == -INFINITY) ? 0.0 : s_z[lane] * (double)exp2f(mw - mm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zz += __shfl_xor_sync(0xffffffffu, zz, o);
    if (lane == 0) {
      ws.m[row] = mm;
      ws.z[row] = zz;
    }
  }
}

// Weight of token t in the sampling row: p_t, or max(0, p_t - q_t) for a residual.
struct RowWeights {
  const float* pr;
  const float* qr;
  float pm, qm, inv_zp, inv_zq, inv_t;
  bool resid;
  __device__ __forceinline__ float operator()(int t) const {
    const float pt = exp2f(__ldg(pr + t) * inv_t - pm) * inv_zp;
    if (!resid) return pt;
    return fmaxf(pt - exp2f(__ldg(qr + t) * inv_t - qm) * inv_zq, 0.0f);
  }
};

// (2) Tests and draw.  GS threads per sequence (a warp, or a whole block).
// STAGE (GS = 1024 only): the sampling row's weights are computed once with
// coalesced loads into shared memory, laid out as every thread's contiguous
// vocabulary slice (seg floats at a pitch of seg + 1, so slice reads are free
// of bank conflicts); the slice sums and the walk read them from there.
template <int GS, bool STAGE = false>
__global__ void __launch_bounds__(GS == 32 ? 256 : GS) accept_kernel(
    const float* __restrict__ tgt, const float* __restrict__ drf, const int32_t* __restrict__ tokens,
    const float* __restrict__ u_acc, const float* __restrict__ u_res, int B, int gamma, int V, float inv_t,
    double inv_t_d, NormWs ws, int32_t* __restrict__ n_acc, int32_t* __restrict__ next_token,
    int32_t* __restrict__ out_tokens) {
  extern __shared__ float s_w[];
  __shared__ float s_ph[32], s_pl[32], s_th, s_tl;
  __shared__ double s_total;
  __shared__ int s_found[32], s_lastv[32];
  __shared__ int s_g, s_nacc;
  pdl_wait();
  const int gid = threadIdx.x % GS;  // thread index inside the sequence's group
  const int b = GS == 32 ? (int)(blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) : (int)blockIdx.x;
  const bool live = b < B;  // (warp groups only) groups past B just follow along
  const int R = 2 * gamma + 1;
  const int lane = threadIdx.x & 31;

  // ---- draft length and the ratio tests (fp64)
  // The group's first warp takes 32 draft positions at a time: lane i loads
  // everything test i needs (all loads in flight together) and decides it; the
  // first position outside the draft and the first rejection come from ballots.
  int nacc = 0, g = 0;
  if (live && gid < 32) {
    g = gamma;
    int first_rej = gamma;
    for (int base = 0; base < gamma; base += 32) {
      const int i = base + gid;
      bool in_draft = false, accept = false;
      if (i < gamma) {
        const int xi = tokens[(size_t)b * gamma + i];
        in_draft = xi >= 0 && xi < V;
        if (in_draft) {
          const double zp = ws.z[(size_t)b * R + i];
          const double zq = ws.z[(size_t)b * R + gamma + 1 + i];
          const double lp =
              (double)tgt[((size_t)b * (gamma + 1) + i) * V + xi] * inv_t_d - (double)ws.m[(size_t)b * R + i];
          const double lq = (double)drf[((size_t)b * gamma + i) * V + xi] * inv_t_d -
                            (double)ws.m[(size_t)b * R + gamma + 1 + i];
          const double ua = (double)u_acc[(size_t)b * gamma + i];
          accept = (exp2(lq) / zq == 0.0) || ua <= exp2(lp - lq) * (zq / zp);
        }
      }
      const unsigned outside = __ballot_sync(0xffffffffu, i < gamma && !in_draft);
      const unsigned rej = __ballot_sync(0xffffffffu, in_draft && !accept);
      if (outside) g = base + __ffs(outside) - 1;
      if (rej) first_rej = base + __ffs(rej) - 1;
      if (outside || rej) break;  // the first of the two ends the tests (warp-uniform)
    }
    // a rejection past the end of the draft is no rejection
    nacc = min(g, first_rej);
  }
  if (GS == 32) {
    g = __shfl_sync(0xffffffffu, g, 0);
    nacc = __shfl_sync(0xffffffffu, nacc, 0);
  } else {
    if (gid == 0) {
      s_g = g;
      s_nacc = nacc;
    }
    __syncthreads();
    g = s_g;
    nacc = s_nacc;
  }

  // ---- the sampling row: residual at the first rejection, else the bonus row
  const bool rejected = nacc < g;
  const int j = nacc;
  const int bb = live ? b : 0;
  RowWeights w;
  w.inv_t = inv_t;
  w.pr = tgt + ((size_t)bb * (gamma + 1) + j) * V;
  w.qr = rejected ? drf + ((size_t)bb * gamma + j) * V : w.pr;
  w.pm = ws.m[(size_t)bb * R + j];
  w.inv_zp = (float)(1.0 / ws.z[(size_t)bb * R + j]);
  w.qm = rejected ? ws.m[(size_t)bb * R + gamma + 1 + j] : 0.0f;
  w.inv_zq = rejected ? (float)(1.0 / ws.z[(size_t)bb * R + gamma + 1 + j]) : 0.0f;
  const double u = live ? (double)u_res[b] : 0.0;
  const int seg = (V + GS - 1) / GS;
  const int t0 = min(V, gid * seg), t1 = min(V, t0 + seg);

  int next = 0;
  for (int attempt = 0; attempt < 2; ++attempt) {
    w.resid = rejected && attempt == 0;
    // slice sum (in index order)
    float run = 0.0f;
    const float* mine = s_w + (size_t)gid * (seg + 1);
    if (STAGE) {
      __syncthreads();  // (attempt 1) every reader of the previous weights is done
      for (int e = gid; e < V; e += GS) {
        const int owner = e / seg;
        s_w[(size_t)owner * (seg + 1) + (e - owner * seg)] = w(e);
      }
      __syncthreads();
      for (int k = 0; k < t1 - t0; ++k) run += mine[k];
    } else {
      for (int t = t0; t < t1; t += kBatch) {
        float v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) v[k] = (t + k < t1) ? w(t + k) : 0.0f;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) run += v[k];
      }
    }
    // Position of this slice in the row's cumulative sum: excl (before it) and
    // total, then whether the crossing u * total falls inside it (gap: how far
    // past excl the crossing lies).  A warp scans in fp64; a block scans
    // exact fp32 pairs (hi + lo, ~44 bits: fp64 is scarce on this part) and
    // one thread forms the crossing in fp64.
    bool holds;
    float gap;
    double total;
    if (GS == 32) {
      double incl = (double)run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      total = __shfl_sync(0xffffffffu, incl, 31);
      const double excl = incl - (double)run;
      const double target = u * total;
      holds = excl <= target && excl + (double)run > target;
      gap = (float)(target - excl);
    } else {
      float ih = run, il = 0.0f;  // inclusive prefix inside the warp, as a pair
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float h2 = __shfl_up_sync(0xffffffffu, ih, o), l2 = __shfl_up_sync(0xffffffffu, il, o);
        if (lane >= o) pair_add(ih, il, h2, l2);
      }
      float eh = __shfl_up_sync(0xffffffffu, ih, 1), el = __shfl_up_sync(0xffffffffu, il, 1);
      if (lane == 0) eh = el = 0.0f;  // exclusive prefix inside the warp
      const int warp = threadIdx.x >> 5, nw = GS / 32;
      __syncthreads();
      if (lane == 31) {
        s_ph[warp] = ih;
        s_pl[warp] = il;
      }
      __syncthreads();
      if (warp == 0) {
        const float vh = lane < nw ? s_ph[lane] : 0.0f, vl = lane < nw ? s_pl[lane] : 0.0f;
        float wh = vh, wl = vl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float h2 = __shfl_up_sync(0xffffffffu, wh, o), l2 = __shfl_up_sync(0xffffffffu, wl, o);
          if (lane >= o) pair_add(wh, wl, h2, l2);
        }
        float xh = __shfl_up_sync(0xffffffffu, wh, 1), xl = __shfl_up_sync(0xffffffffu, wl, 1);
        if (lane == 0) xh = xl = 0.0f;
        __syncwarp();
        if (lane < nw) {
          s_ph[lane] = xh;  // exclusive prefix of warp `lane`
          s_pl[lane] = xl;
        }
        if (lane == 31) {
          const double tot = (double)wh + (double)wl;
          const double tgt = u * tot;
          s_total = tot;
          s_th = (float)tgt;
          s_tl = (float)(tgt - (double)(float)tgt);
        }
      }
      __syncthreads();
      total = s_total;
      float xh = s_ph[warp], xl = s_pl[warp];
      pair_add(xh, xl, eh, el);  // excl = the warp's prefix + the prefix inside the warp
      // gap = target - excl, to fp32 rounding of a value below the slice sum
      gap = ((s_th - xh) + (s_tl - xl));
      holds = gap >= 0.0f && run > gap;
    }
    if (!(total > 0.0)) {
      if (w.resid) continue;  // p == q: the residual is empty, draw from p_j instead
      break;                  // (not reachable for finite logits)
    }
    // the slice holding the crossing walks it again, in the same order
    int found = 0x7fffffff, last = -1;
    if (holds) {
      float r2 = 0.0f;
      for (int t = t0; t < t1; ++t) {
        r2 += STAGE ? mine[t - t0] : w(t);
        if (r2 > gap) {
          found = t;
          break;
        }
      }
    }
    // rounding can leave no crossing: then the last index with positive weight
    bool any;
    if (GS == 32) {
      any = __any_sync(0xffffffffu, found != 0x7fffffff);
    } else {
      any = __syncthreads_or(found != 0x7fffffff);
    }
    if (!any) {
      for (int t = t0; t < t1; ++t)
        if ((STAGE ? mine[t - t0] : w(t)) > 0.0f) last = t;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
      last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    }
    if (GS != 32) {
      const int warp = threadIdx.x >> 5, nw = GS / 32;
      __syncthreads();
      if (lane == 0) {
        s_found[warp] = found;
        s_lastv[warp] = last;
      }
      __syncthreads();
      for (int k = 0; k < nw; ++k) {
        found = min(found, s_found[k]);
        last = max(last, s_lastv[k]);
      }
    }
    next = found != 0x7fffffff ? found : (last >= 0 ? last : 0);
    break;
  }

  if (live) {
    if (gid == 0) {
      n_acc[b] = nacc;
      next_token[b] = next;
    }
    if (out_tokens) {
      const int32_t* x = tokens + (size_t)b * gamma;
      for (int c = gid; c <= gamma; c += GS) {
        int v = -1;
        if (c < nacc)
          v = x[c];
        else if (c == nacc)
          v = next;
        out_tokens[(size_t)b * (gamma + 1) + c] = v;
      }
    }
  }
}

size_t norm_bytes(int B, int gamma) {
  const size_t rows = (size_t)B * (2 * gamma + 1);
  return align_up(rows * sizeof(float), 256) + rows * sizeof(double);
}

// ---------------------------------------------------------------------------
// Tree form (candidates with parent links).  The same rule applied to the
// children of a node one at a time, in index order: a child passes when
// u <= p'(x) / q(x); a child that fails turns p' into max(0, p' - q)
// normalised and the next sibling is tested; a child that passes restarts
// the walk at it with the verifier row after it; a node with no child left
// draws the next token from p'.
//
// One block per sequence.  Warp 0 walks the tree (next child by ballot over
// the parent links, fp64 ratio tests from the normalisers, as in the chain
// kernel); only a rejection needs the whole block, for a pass over the
// vocabulary that forms the residual and sums it.  The final draw scans the
// row holding p' with the chain kernel's fp32-pair scan.
struct TreeParams {
  const float* tgt;      // [B, T+1, V]
  const float* drf;      // [B, T, V]
  const int32_t* tokens;  // [B, T]
  const int32_t* parent;  // [B, T]
  const float* u_acc;    // [B, T]
  const float* u_res;    // [B]
  int T, V, Vpad;
  float inv_t;
  double inv_t_d;
  NormWs ws;    // [B, 2T+1]
  float* wbuf;  // [B, 2, Vpad]
  int32_t* n_acc;
  int32_t* next_token;
  int32_t* out_tokens;  // [B, T+1] or null
  int32_t* acc_nodes;   // [B, T] or null
};

// Index-order inverse CDF over the weights of tokens [0, V) with 1024 threads
// (every thread of the block): thread g owns the contiguous slice of tokens
// [g * seg, (g + 1) * seg), stored at w[g * pitch + k] (pitch = seg: a plain
// row; seg + 1: the bank-conflict-free shared-memory layout); the slice sums
// are scanned as exact fp32 pairs, one thread forms the crossing u * total in
// fp64 and the slice holding it is walked again.  Returns the drawn index (all
// threads); the last index with positive weight if rounding leaves no crossing.
__device__ int block_inverse_cdf(const float* __restrict__ w, int V, int pitch, double u) {
  constexpr int GS = kBlockSeq;
  __shared__ float s_ph[32], s_pl[32], s_th, s_tl;
  __shared__ int s_found[32], s_lastv[32];
  const int gid = threadIdx.x, lane = gid & 31, warp = gid >> 5, nw = GS / 32;
  const int seg = (V + GS - 1) / GS;
  const int t0 = min(V, gid * seg), t1 = min(V, t0 + seg);
  const float* mine = w + (size_t)gid * pitch - t0;  // mine[t]: the weight of token t of this slice
  float run = 0.0f;
  for (int t = t0; t < t1; ++t) run += mine[t];
  float ih = run, il = 0.0f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float h2 = __shfl_up_sync(0xffffffffu, ih, o), l2 = __shfl_up_sync(0xffffffffu, il, o);
    if (lane >= o) pair_add(ih, il, h2, l2);
  }
  float eh = __shfl_up_sync(0xffffffffu, ih, 1), el = __shfl_up_sync(0xffffffffu, il, 1);
  if (lane == 0) eh = el = 0.0f;
  __syncthreads();
  if (lane == 31) {
    s_ph[warp] = ih;
    s_pl[warp] = il;
  }
  __syncthreads();
  if (warp == 0) {
    const float vh = lane < nw ? s_ph[lane] : 0.0f, vl = lane < nw ? s_pl[lane] : 0.0f;
    float wh = vh, wl = vl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float h2 = __shfl_up_sync(0xffffffffu, wh, o), l2 = __shfl_up_sync(0xffffffffu, wl, o);
      if (lane >= o) pair_add(wh, wl, h2, l2);
    }
    float xh = __shfl_up_sync(0xffffffffu, wh, 1), xl = __shfl_up_sync(0xffffffffu, wl, 1);
    if (lane == 0) xh = xl = 0.0f;
    __syncwarp();
    if (lane < nw) {
      s_ph[lane] = xh;
      s_pl[lane] = xl;
    }
    if (lane == 31) {
      const double tgt = u * ((double)wh + (double)wl);
      s_th = (float)tgt;
      s_tl = (float)(tgt - (double)(float)tgt);
    }
  }
  __syncthreads();
  float xh = s_ph[warp], xl = s_pl[warp];
  pair_add(xh, xl, eh, el);
  const float gap = (s_th - xh) + (s_tl - xl);
  const bool holds = gap >= 0.0f && run > gap;
  int found = 0x7fffffff, last = -1;
  if (holds) {
    float r2 = 0.0f;
    for (int t = t0; t < t1; ++t) {
      r2 += mine[t];
      if (r2 > gap) {
        found = t;
        break;
      }
    }
  }
  if (!__syncthreads_or(found != 0x7fffffff)) {
    for (int t = t0; t < t1; ++t)
      if (mine[t] > 0.0f) last = t;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
    last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  }
  __syncthreads();
  if (lane == 0) {
    s_found[warp] = found;
    s_lastv[warp] = last;
  }
  __syncthreads();
  for (int k = 0; k < nw; ++k) {
    found = min(found, s_found[k]);
    last = max(last, s_lastv[k]);
  }
  return found != 0x7fffffff ? found : (last >= 0 ? last : 0);
}

// Parent of candidate j as the tree calls read it (a link outside [-1, j) is -1).
__device__ __forceinline__ int tree_parent(const int32_t* par, int j) {
  const int pj = par[j];
  return (pj >= -1 && pj < j) ? pj : -1;
}

// SMEM: p' after a rejection is held in dynamic shared memory (one row, the
// bank-conflict-free slice layout of the chain kernel's staging: token e at
// (e / seg) * (seg + 1) + e % seg); each rejection then takes two passes, the
// residual's sum and, only when that sum is positive, its in-place write, so
// an all-zero residual still leaves p' as it was.  Otherwise (vocabularies
// too large for shared memory) p' lives in two workspace rows, the residual
// written into the row that does not hold p'.
template <bool SMEM>
__global__ void __launch_bounds__(kBlockSeq) tree_accept_kernel(TreeParams p) {
  extern __shared__ float s_w[];
  __shared__ int s_node, s_staged, s_rej, s_depth;
  __shared__ double s_Z, s_part[32];
  pdl_wait();
  const int b = blockIdx.x, T = p.T, V = p.V, R = 2 * T + 1;
  const int gid = threadIdx.x, lane = gid & 31, warp = gid >> 5;
  const int seg = (V + kBlockSeq - 1) / kBlockSeq;
  const int32_t* tok = p.tokens + (size_t)b * T;
  const int32_t* par = p.parent + (size_t)b * T;
  float* buf = SMEM ? s_w : p.wbuf + (size_t)b * 2 * p.Vpad;
  // where token e of the p' row `which` is stored (e / seg as a multiply-high
  // by the rounded-up reciprocal of seg, exact for e < 2^32 / seg; seg = 1,
  // whose reciprocal 2^32 does not fit 32 bits, is the identity)
  const uint32_t recip = seg > 1 ? (uint32_t)((0xffffffffull + (uint32_t)seg) / (uint32_t)seg) : 0u;
  auto at = [&](int which, int e) -> size_t {
    if (SMEM) {
      const int o = seg > 1 ? (int)__umulhi((uint32_t)e, recip) : e;
      return (size_t)o * (seg + 1) + (e - o * seg);
    }
    return (size_t)which * p.Vpad + e;
  };
  // Walk state, kept by thread 0 and published for the block: the current
  // node (-1: the prefix); which row holds p' (-1: p' is the verifier row
  // after the node) and its sum.
  if (gid == 0) {
    s_node = -1;
    s_staged = -1;
    s_depth = 0;
    s_Z = 0.0;
  }
  __syncthreads();
  int last = -1;  // warp 0: candidates up to here have been visited
  while (true) {
    if (warp == 0) {
      int node = s_node, staged = s_staged, depth = s_depth;
      const double Z = s_Z;
      int rej = -1;
      while (true) {
        // next child of `node` after `last`, in index order
        int c = -1;
        for (int base = last + 1; base < T; base += 32) {
          const int j = base + lane;
          bool ok = false;
          if (j < T) {
            const int x = tok[j];
            ok = x >= 0 && x < V && tree_parent(par, j) == node;
          }
          const unsigned ball = __ballot_sync(0xffffffffu, ok);
          if (ball) {
            c = base + __ffs(ball) - 1;
            break;
          }
        }
        if (c < 0) break;
        last = c;
        bool accept = false;
        if (lane == 0) {
          const int x = tok[c];
          const double lq = (double)p.drf[((size_t)b * T + c) * V + x] * p.inv_t_d -
                            (double)p.ws.m[(size_t)b * R + T + 1 + c];
          const double zq = p.ws.z[(size_t)b * R + T + 1 + c];
          const double ua = (double)p.u_acc[(size_t)b * T + c];
          if (staged < 0) {
            const int row = node + 1;
            const double lp = (double)p.tgt[((size_t)b * (T + 1) + row) * V + x] * p.inv_t_d -
                              (double)p.ws.m[(size_t)b * R + row];
            const double zp = p.ws.z[(size_t)b * R + row];
            accept = (exp2(lq) / zq == 0.0) || ua <= exp2(lp - lq) * (zq / zp);
          } else {
            const double wx = (double)buf[at(staged, x)];
            accept = (exp2(lq) / zq == 0.0) || ua <= (wx / Z) * zq / exp2(lq);
          }
          if (accept) {
            if (p.out_tokens) p.out_tokens[(size_t)b * (T + 1) + depth] = x;
            if (p.acc_nodes) p.acc_nodes[(size_t)b * T + depth] = c;
          }
        }
        accept = __shfl_sync(0xffffffffu, accept, 0);
        if (!accept) {
          rej = c;
          break;
        }
        node = c;
        staged = -1;
        ++depth;
      }
      if (lane == 0) {
        s_node = node;
        s_staged = staged;
        s_depth = depth;
        s_rej = rej;
      }
    }
    __syncthreads();
    const int rej = s_rej;
    if (rej < 0) break;
    // ---- residual of p' against the rejected candidate's drafter row
    const int node = s_node, staged = s_staged;
    const int dst = SMEM ? 0 : (staged == 0 ? 1 : 0);
    const float* qr = p.drf + ((size_t)b * T + rej) * V;
    const float qm = p.ws.m[(size_t)b * R + T + 1 + rej];
    const float inv_zq = (float)(1.0 / p.ws.z[(size_t)b * R + T + 1 + rej]);
    const float* pr = p.tgt + ((size_t)b * (T + 1) + node + 1) * V;
    const float pm = p.ws.m[(size_t)b * R + node + 1];
    const float inv_zp = (float)(1.0 / p.ws.z[(size_t)b * R + node + 1]);
    const float inv_Z = staged >= 0 ? (float)(1.0 / s_Z) : 0.0f;
    auto resid = [&](int t) {
      const float cur = staged >= 0 ? buf[at(staged, t)] * inv_Z : exp2f(__ldg(pr + t) * p.inv_t - pm) * inv_zp;
      return fmaxf(cur - exp2f(__ldg(qr + t) * p.inv_t - qm) * inv_zq, 0.0f);
    };
    double part = 0.0;
    for (int t = gid; t < V; t += kBlockSeq) {
      const float r = resid(t);
      if (!SMEM) buf[at(dst, t)] = r;
      part += (double)r;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) s_part[warp] = part;
    __syncthreads();
    double z = 0.0;
    for (int w = 0; w < kBlockSeq / 32; ++w) z += s_part[w];
    if (SMEM && z > 0.0) {
      // the same residual again, now written over p' (each token by one thread)
      for (int t = gid; t < V; t += kBlockSeq) {
        const float r = resid(t);
        buf[at(0, t)] = r;
      }
    }
    __syncthreads();
    if (gid == 0 && z > 0.0) {  // an all-zero residual leaves p' as it was
      s_staged = dst;
      s_Z = z;
    }
    __syncthreads();
  }
  // ---- the draw: p' into a row if it is still a verifier row
  const int node = s_node, depth = s_depth;
  int staged = s_staged;
  if (staged < 0) {
    const float* pr = p.tgt + ((size_t)b * (T + 1) + node + 1) * V;
    const float pm = p.ws.m[(size_t)b * R + node + 1];
    const float inv_zp = (float)(1.0 / p.ws.z[(size_t)b * R + node + 1]);
    for (int t = gid; t < V; t += kBlockSeq) buf[at(0, t)] = exp2f(__ldg(pr + t) * p.inv_t - pm) * inv_zp;
    staged = 0;
    __syncthreads();
  }
  const int next = SMEM ? block_inverse_cdf(buf, V, seg + 1, (double)p.u_res[b])
                        : block_inverse_cdf(buf + (size_t)staged * p.Vpad, V, seg, (double)p.u_res[b]);
  if (gid == 0) {
    p.n_acc[b] = depth;
    p.next_token[b] = next;
  }
  if (p.out_tokens)
    for (int c = depth + gid; c <= T; c += kBlockSeq) p.out_tokens[(size_t)b * (T + 1) + c] = c == depth ? next : -1;
  if (p.acc_nodes)
    for (int c = depth + gid; c < T; c += kBlockSeq) p.acc_nodes[(size_t)b * T + c] = -1;
}

size_t tree_bytes(int B, int T, int V) {
  return align_up(norm_bytes(B, T), 256) + (size_t)B * 2 * align_up((size_t)V, 64) * sizeof(float);
}


}  // namespace
}  // namespace tf

extern "C" size_t tf_spec_accept_workspace(int B, int gamma) {
  if (B <= 0 || gamma < 0) return 0;
  return tf::norm_bytes(B, gamma);
}

extern "C" tf_status tf_spec_accept(const float* tgt_logits, const float* drf_logits, const int32_t* drf_tokens,
                                    const float* u_acc, const float* u_res, int B, int gamma, int V,
                                    float temperature, int32_t* n_acc, int32_t* next_token, int32_t* out_tokens,
                                    void* ws, size_t ws_bytes, tf_stream_t stream) {
  using namespace tf;
  if (!tgt_logits || !u_res || !n_acc || !next_token) return TF_ERR_INVALID_ARG;
  if (gamma > 0 && (!drf_logits || !drf_tokens || !u_acc)) return TF_ERR_INVALID_ARG;
  if (B < 0 || gamma < 0 || V < 1 || !(temperature > 0.0f)) return TF_ERR_INVALID_ARG;
  if (B == 0) return TF_OK;
  if (!ws || ws_bytes < norm_bytes(B, gamma) || !aligned16(ws)) return TF_ERR_WORKSPACE;
  const long long rows = (long long)B * (2 * gamma + 1);
  if (rows >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
  NormWs nws;
  nws.m = static_cast<float*>(ws);
  nws.z = reinterpret_cast<double*>(static_cast<char*>(ws) + align_up((size_t)rows * sizeof(float), 256));
  const double inv_t_d = 1.4426950408889634 / (double)temperature;  // log2(e) / temperature
  const float inv_t = (float)inv_t_d;
  cudaError_t e;
  if (V <= kSmallV) {
    e = launch_pdl(row_norm_kernel<true>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, stream, tgt_logits,
                   drf_logits, B, gamma, V, inv_t, nws);
    if (e == cudaSuccess)
      e = launch_pdl(accept_kernel<32>, dim3((unsigned)((B + 7) / 8)), dim3(256), 0, stream, tgt_logits, drf_logits,
                     drf_tokens, u_acc, u_res, B, gamma, V, inv_t, inv_t_d, nws, n_acc, next_token, out_tokens);
  } else {
    e = launch_pdl(row_norm_kernel<false>, dim3((unsigned)rows), dim3(kBlockRow), 0, stream, tgt_logits, drf_logits,
                   B, gamma, V, inv_t, nws);
    const int seg = (V + kBlockSeq - 1) / kBlockSeq;
    const size_t stage_bytes = (size_t)kBlockSeq * (seg + 1) * sizeof(float);
    if (e == cudaSuccess && stage_bytes <= kMaxStageBytes) {
      static DeviceCache configured;
      if (!configured.get([] {
            return cudaFuncSetAttribute(accept_kernel<kBlockSeq, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kMaxStageBytes) == cudaSuccess;
          }))
        return TF_ERR_CUDA;
      e = launch_pdl(accept_kernel<kBlockSeq, true>, dim3(B), dim3(kBlockSeq), stage_bytes, stream, tgt_logits,
                     drf_logits, drf_tokens, u_acc, u_res, B, gamma, V, inv_t, inv_t_d, nws, n_acc, next_token,
                     out_tokens);
    } else if (e == cudaSuccess) {
      e = launch_pdl(accept_kernel<kBlockSeq>, dim3(B), dim3(kBlockSeq), 0, stream, tgt_logits, drf_logits,
                     drf_tokens, u_acc, u_res, B, gamma, V, inv_t, inv_t_d, nws, n_acc, next_token, out_tokens);
    }
  }
  return e == cudaSuccess ? launch_status() : TF_ERR_CUDA;
}

extern "C" size_t tf_spec_accept_tree_workspace(int B, int T, int V) {
  if (B <= 0 || T < 0 || V < 1) return 0;
  return tf::tree_bytes(B, T, V);
}

extern "C" tf_status tf_spec_accept_tree(const float* tgt_logits, const float* drf_logits, const int32_t* drf_tokens,
                                         const int32_t* parent, const float* u_acc, const float* u_res, int B, int T,
                                         int V, float temperature, int32_t* n_acc, int32_t* next_token,
                                         int32_t* out_tokens, int32_t* acc_nodes, void* ws, size_t ws_bytes,
                                         tf_stream_t stream) {
  using namespace tf;
  if (!tgt_logits || !u_res || !n_acc || !next_token) return TF_ERR_INVALID_ARG;
  if (T > 0 && (!drf_logits || !drf_tokens || !parent || !u_acc)) return TF_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || V < 1 || !(temperature > 0.0f)) return TF_ERR_INVALID_ARG;
  if (B == 0) return TF_OK;
  if (!ws || ws_bytes < tree_bytes(B, T, V) || !aligned16(ws)) return TF_ERR_WORKSPACE;
  const long long rows = (long long)B * (2 * T + 1);
  if (rows >= (1ll << 31) || (long long)B * (T + 1) * V >= (1ll << 40)) return TF_ERR_UNSUPPORTED;
  NormWs nws;
  nws.m = static_cast<float*>(ws);
  nws.z = reinterpret_cast<double*>(static_cast<char*>(ws) + align_up((size_t)rows * sizeof(float), 256));
  TreeParams tp;
  tp.tgt = tgt_logits;
  tp.drf = drf_logits;
  tp.tokens = drf_tokens;
  tp.parent = parent;
  tp.u_acc = u_acc;
  tp.u_res = u_res;
  tp.T = T;
  tp.V = V;
  tp.Vpad = (int)align_up((size_t)V, 64);
  tp.inv_t_d = 1.4426950408889634 / (double)temperature;  // log2(e) / temperature
  tp.inv_t = (float)tp.inv_t_d;
  tp.ws = nws;
  tp.wbuf = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(norm_bytes(B, T), 256));
  tp.n_acc = n_acc;
  tp.next_token = next_token;
  tp.out_tokens = out_tokens;
  tp.acc_nodes = acc_nodes;
  cudaError_t e;
  if (V <= kSmallV)
    e = launch_pdl(row_norm_kernel<true>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, (cudaStream_t)stream,
                   tgt_logits, drf_logits, B, T, V, tp.inv_t, nws);
  else
    e = launch_pdl(row_norm_kernel<false>, dim3((unsigned)rows), dim3(kBlockRow), 0, (cudaStream_t)stream,
                   tgt_logits, drf_logits, B, T, V, tp.inv_t, nws);
  const int seg = (V + kBlockSeq - 1) / kBlockSeq;
  const size_t stage_bytes = (size_t)kBlockSeq * (seg + 1) * sizeof(float);
  if (e == cudaSuccess && stage_bytes <= kMaxStageBytes) {
    static DeviceCache configured;
    if (!configured.get([] {
          return cudaFuncSetAttribute(tree_accept_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kMaxStageBytes) == cudaSuccess;
        }))
      return TF_ERR_CUDA;
    e = launch_pdl(tree_accept_kernel<true>, dim3(B), dim3(kBlockSeq), stage_bytes, (cudaStream_t)stream, tp);
  } else if (e == cudaSuccess) {
    e = launch_pdl(tree_accept_kernel<false>, dim3(B), dim3(kBlockSeq), 0, (cudaStream_t)stream, tp);
  }
  return e == cudaSuccess ? launch_status() : TF_ERR_CUDA;
}
