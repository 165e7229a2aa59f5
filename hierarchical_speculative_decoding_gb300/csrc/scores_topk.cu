// a2 + a3 -- chunk scores and top-k selection for the Force 2 retrieval drafter.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": Force 2 keeps a small top-k subset of the KV blocks, chosen by
// key-query similarity.  Score of chunk c for (sequence b, KV head g):
//   s = (sum of the group's query heads) . M[b, g, c, :]   (fp32 accumulation)
// Selection: the kc largest scores, equal scores to the lower chunk id, ids
// written in ascending order.
//
// Design: one kernel.  The (b, g) units are few (32 at batch 1) while each
// holds up to ~16K chunks, so every unit is split over several CTAs that stream
// the chunk means (a half-warp per 256-byte mean row, 16-byte loads) and write
// fp32 scores to the workspace.  The last CTA of a unit to finish (an atomic
// ticket; no CTA ever waits) runs an exact radix select on order-preserving
// uint32 keys (11 + 11 + 10 bits), then compacts the winners in id order with a
// block-wide scan, so ties resolve to the lower id without any sort.
#include "tf_common.cuh"

namespace tf {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

inline size_t tickets_bytes(int units) { return align_up((size_t)units * sizeof(int), 256); }

// Exclusive block scan of two 0/1 flags; returns the block totals.
__device__ __forceinline__ void block_scan2(bool a, bool b, int& a_ex, int& b_ex, int& a_tot, int& b_tot,
                                            int* sa, int* sb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned ba = __ballot_sync(0xffffffffu, a), bb = __ballot_sync(0xffffffffu, b);
  const unsigned below = (1u << lane) - 1u;
  if (lane == 0) {
    sa[warp] = __popc(ba);
    sb[warp] = __popc(bb);
  }
  __syncthreads();
  int pa = 0, pb = 0, ta = 0, tb = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int xa = sa[w], xb = sb[w];
    if (w < warp) { pa += xa; pb += xb; }
    ta += xa;
    tb += xb;
  }
  a_ex = pa + __popc(ba & below);
  b_ex = pb + __popc(bb & below);
  a_tot = ta;
  b_tot = tb;
  __syncthreads();
}

// Radix-select the kc-th largest key among keys[0, C) (C > kc); returns the
// threshold key and how many keys equal to it are to be taken.
__device__ void radix_select(const float* __restrict__ scores, int C, int kc, unsigned* hist,
                             uint32_t& thresh, int& take_eq) {
  __shared__ int s_bin, s_krem;
  uint32_t prefix = 0, pmask = 0;
  int krem = kc;
  const int shifts[3] = {21, 10, 0};
  const int nbits[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const int nb = 1 << nbits[pass];
    const uint32_t mask = (uint32_t)nb - 1u;
    for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < C; c += kThreads) {
      const uint32_t key = score_key(__ldcg(scores + c));
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & mask], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const int seg = nb / 32;
      const int top = nb - lane * seg;  // lane 0 owns the highest bins
      int segsum = 0;
      for (int i = top - seg; i < top; ++i) segsum += (int)hist[i];
      int incl = segsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = incl - segsum;
      if (excl < krem && krem <= incl) {
        int run = excl;
        for (int i = top - 1; i >= top - seg; --i) {
          const int h = (int)hist[i];
          if (run + h >= krem) {
            s_bin = i;
            s_krem = krem - run;
            break;
          }
          run += h;
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)s_bin << shift;
    pmask |= mask << shift;
    krem = s_krem;
    __syncthreads();
  }
  thresh = prefix;
  take_eq = krem;
}

__global__ void __launch_bounds__(kThreads) scores_topk_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ M, const int32_t* __restrict__ seq_lens,
    int Hq, int Hkv, int Lmax, int kc, int splits, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
    float* __restrict__ s_cut, int* __restrict__ tickets, float* __restrict__ scores_ws) {
  __shared__ float qs[kHeadDim];
  __shared__ unsigned hist[2048];
  __shared__ int scan_a[kWarps], scan_b[kWarps];
  __shared__ int s_last;
  __shared__ float s_min[kWarps];

  const int unit = blockIdx.y;
  const int b = unit / Hkv, g = unit % Hkv;
  const int G = Hq / Hkv;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;
  const int L = clamp_len(seq_lens[b], Lmax);
  const int C = (L + kChunk - 1) / kChunk;
  float* scores = scores_ws + (size_t)unit * Cmax;

  if (threadIdx.x < kHeadDim) {
    float s = 0.0f;
    for (int h = 0; h < G; ++h)
      s += __uint_as_float((uint32_t)q[((size_t)b * Hq + (size_t)g * G + h) * kHeadDim + threadIdx.x] << 16);
    qs[threadIdx.x] = s;
  }
  __syncthreads();

  // ---- scoring: this CTA's slice of the unit's chunks
  const int per = (C + splits - 1) / splits;
  const int c0 = blockIdx.x * per;
  const int c1 = min(C, c0 + per);
  const int half = (threadIdx.x >> 4) & 1, l16 = threadIdx.x & 15, wid = threadIdx.x >> 5;
  float qv[8];
#pragma unroll
  for (int d = 0; d < 8; ++d) qv[d] = qs[l16 * 8 + d];
  const uint16_t* Mu = M + (size_t)unit * Cmax * kHeadDim + l16 * 8;
  constexpr int kHalfWarps = kThreads / 16;
  // The loop bound is warp-uniform (the shuffles below need the whole warp);
  // each half-warp owns chunk base + half + u * kHalfWarps.
  for (int base = c0 + 2 * wid; base < c1; base += kHalfWarps * kUnroll) {
    const int cb = base + half;
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = cb + u * kHalfWarps;
      v[u] = (c < c1) ? ld_stream16(Mu + (size_t)c * kHeadDim) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float f[8];
      unpack8(v[u], f);
      float s = 0.0f;
#pragma unroll
      for (int d = 0; d < 8; ++d) s = fmaf(qv[d], f[d], s);
      s += __shfl_xor_sync(0xffffffffu, s, 8);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      const int c = cb + u * kHalfWarps;
      if (l16 == 0 && c < c1) scores[c] = s;
    }
  }

  // ---- ticket: the last CTA of this unit selects
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&tickets[unit], 1) == splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  int32_t* out = idx + (size_t)unit * kc;
  if (C <= kc) {
    float mn = INFINITY;
    for (int c = threadIdx.x; c < kc; c += kThreads) {
      out[c] = (c < C) ? c : -1;
      if (c < C) mn = fminf(mn, __ldcg(scores + c));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    if ((threadIdx.x & 31) == 0) s_min[threadIdx.x >> 5] = mn;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = INFINITY;
      for (int w = 0; w < kWarps; ++w) m = fminf(m, s_min[w]);
      n_sel[unit] = C;
      if (s_cut) s_cut[unit] = (C > 0) ? m : -INFINITY;
      tickets[unit] = 0;
    }
    return;
  }

  uint32_t T;
  int take_eq;
  radix_select(scores, C, kc, hist, T, take_eq);

  int run_out = 0, run_eq = 0;
  for (int base = 0; base < C; base += kThreads) {
    const int c = base + threadIdx.x;
    const uint32_t key = (c < C) ? score_key(__ldcg(scores + c)) : 0u;
    const bool gt = (c < C) && key > T;
    const bool eq = (c < C) && key == T;
    int eq_ex, dummy_ex, eq_tot, dummy_tot;
    block_scan2(eq, false, eq_ex, dummy_ex, eq_tot, dummy_tot, scan_a, scan_b);
    const bool sel = gt || (eq && (run_eq + eq_ex) < take_eq);
    int sel_ex, sel_tot;
    block_scan2(sel, false, sel_ex, dummy_ex, sel_tot, dummy_tot, scan_a, scan_b);
    if (sel && run_out + sel_ex < kc) out[run_out + sel_ex] = c;
    run_out += sel_tot;
    run_eq += eq_tot;
  }
  if (threadIdx.x == 0) {
    n_sel[unit] = kc;
    if (s_cut) s_cut[unit] = key_score(T);
    tickets[unit] = 0;
  }
}

}  // namespace
}  // namespace tf

namespace {
int scores_splits(int units, int Cmax) {
  const int target = tf::num_sms() * 2;
  int s = (target + units - 1) / units;
  const int max_s = (Cmax + 63) / 64;
  if (s > max_s) s = max_s;
  return s < 1 ? 1 : s;
}
}  // namespace

extern "C" size_t tf_chunk_scores_topk_workspace(int B, int Hkv, int Lmax, int chunk) {
  if (B <= 0 || Hkv <= 0 || Lmax <= 0 || chunk != tf::kChunk) return 0;
  const size_t units = (size_t)B * Hkv;
  const size_t Cmax = (size_t)(Lmax + chunk - 1) / chunk;
  return tf::tickets_bytes((int)units) + units * Cmax * sizeof(float);
}

extern "C" tf_status tf_chunk_scores_topk(const uint16_t* q, const uint16_t* M, const int32_t* seq_lens, int B,
                                          int Hq, int Hkv, int Lmax, int D, int chunk, int kc, int32_t* idx,
                                          int32_t* n_sel, float* s_cut, void* ws, size_t ws_bytes,
                                          tf_stream_t stream) {
  using namespace tf;
  if (!q || !M || !seq_lens || !idx || !n_sel) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || kc <= 0 || Hq % Hkv != 0) return TF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(M)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  const size_t need = tf_chunk_scores_topk_workspace(B, Hkv, Lmax, chunk);
  if (!ws || ws_bytes < need || !aligned16(ws)) return TF_ERR_WORKSPACE;
  const int units = B * Hkv;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;
  const int splits = scores_splits(units, Cmax);
  int* tickets = static_cast<int*>(ws);
  float* scores = reinterpret_cast<float*>(static_cast<char*>(ws) + tickets_bytes(units));
  dim3 grid(splits, units);
  scores_topk_kernel<<<grid, kThreads, 0, stream>>>(q, M, seq_lens, Hq, Hkv, Lmax, kc, splits, idx, n_sel, s_cut,
                                                    tickets, scores);
  return launch_status();
}
