// a2 + a3 building blocks -- chunk scoring and cluster-wide top-k selection.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": Force 2 keeps a small top-k subset of the KV blocks, chosen by
// key-query similarity.  Score of chunk c for (sequence b, KV head g):
//   s = (sum of the group's query heads) . M[b, g, c, :]   (fp32 accumulation)
// Selection: the kc largest scores, equal scores to the lower chunk id.
//
// One thread-block cluster of S <= 8 CTAs serves one (b, g) unit; CTA r owns
// the r-th contiguous slice of the unit's chunks and keeps its scores in shared
// memory as order-preserving uint32 keys with a histogram of their top 11 bits.
// The cut is found on the whole cluster through distributed shared memory: the
// S histograms are summed on every CTA and give the bin b1 holding the kc-th
// largest key; each CTA publishes its keys of that bin and every CTA gathers
// them and resolves the remaining 21 bits by itself (a rare overflow of the
// candidate buffer falls back to two more cluster histogram rounds).  Every
// key in a bin above b1 is selected, which callers can act on before the cut
// is final; the steps after round 1 can run on a group of eight warps while
// the rest of the CTA does other work.  Used by the top-k call and by the fused
// retrieval-draft call.
#pragma once

#include "sm100_ptx.cuh"
#include "tf_common.cuh"

namespace tf {
namespace topk {

using namespace sm100;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 6;
constexpr int kMaxCluster = 16;         // cluster sizes above 8 need the non-portable opt-in
constexpr int kMaxPortableCluster = 8;
constexpr int kMaxSliceKeys = 16384;  // keys per CTA held in shared memory (64 KB)

// Shared-memory arrays of the selection.  hist*, tot 16-byte aligned.
struct Arrays {
  uint32_t* keys;   // [n] this CTA's score keys
  uint32_t* hist1;  // [2048] top 11 key bits of this slice (read by the cluster)
  uint32_t* hist2;  // [2048]
  uint32_t* hist3;  // [1024]
  uint32_t* tot;    // [2048] cluster sums
  uint32_t* cand;   // [cap] this CTA's keys of bin b1 (read by the cluster)
  uint32_t* gcand;  // [cap] the cluster's keys of bin b1
  int cap;
};

// The cut: keys > T are selected, and of the keys == T the first take_eq in
// chunk-id order over the cluster.
struct Cut {
  uint32_t b1;   // top 11 bits of T
  uint32_t T;
  int take_eq;
  int cta_eq;    // keys == T in the CTAs before this one
  int cta_sel;   // selected chunks in the CTAs before this one
};

__device__ __forceinline__ void zero_hists(const Arrays& a) {
  for (int i = threadIdx.x; i < 2048; i += kThreads) {
    a.hist1[i] = 0;
    a.hist2[i] = 0;
  }
  for (int i = threadIdx.x; i < 1024; i += kThreads) a.hist3[i] = 0;
}

// Barriers for the group of threads running a step: the whole CTA, or warps
// 0..7 on named barrier 1 while the other warps do something else.
struct CtaBar {
  static constexpr int kNT = kThreads;
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
struct Warps0to7Bar {
  static constexpr int kNT = 256;
  __device__ __forceinline__ void operator()() const { asm volatile("bar.sync 1, 256;" ::: "memory"); }
};

// Thread t of the group owns nb / NT bins of h (thread 0 the highest); find the
// bin holding the krem-th largest key.  All threads of the group; result in
// s_bin / s_krem; s_wsum holds NT / 32 ints.
template <class Bar>
__device__ __forceinline__ void find_bin(const uint32_t* h, int nb, int krem, int* s_wsum, int* s_bin, int* s_krem,
                                         Bar bar) {
  constexpr int NT = Bar::kNT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k = nb / NT;
  const int top = nb - (int)threadIdx.x * k;
  int segsum = 0;
  for (int i = top - k; i < top; ++i) segsum += (int)h[i];
  int incl = segsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  bar();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
  incl += wbase;
  const int excl = incl - segsum;
  if (excl < krem && krem <= incl) {
    int run = excl;
    for (int i = top - 1; i >= top - k; --i) {
      const int c = (int)h[i];
      if (run + c >= krem) {
        *s_bin = i;
        *s_krem = krem - run;
        break;
      }
      run += c;
    }
  }
  bar();
}

// tot[i] = sum over the cluster's CTAs of their local[i], i < nb (nb a multiple
// of 4, arrays 16-byte aligned): 16-byte remote loads, all ranks in flight.
__device__ __forceinline__ void cluster_sum(const uint32_t* local, uint32_t* tot, int nb, int S) {
  for (int i = 4 * threadIdx.x; i < nb; i += 4 * kThreads) {
    uint4 t = make_uint4(0, 0, 0, 0);
    for (int r0 = 0; r0 < S; r0 += 8) {  // eight ranks in flight at a time
      uint4 v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        v[r] = r0 + r < S ? dsmem_ld_v4(local + i, (uint32_t)(r0 + r)) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        t.x += v[r].x;
        t.y += v[r].y;
        t.z += v[r].z;
        t.w += v[r].w;
      }
    }
    *reinterpret_cast<uint4*>(tot + i) = t;
  }
  __syncthreads();
}

// Scores of chunks [c0, c1) of one unit into keys[c - c0] and hist1.  qs: the
// group's summed query (128 floats in shared memory); Mu: the unit's means
// (cmax rows).  A half-warp reads one 256-byte mean row with 16-byte loads, U
// rows in flight per half-warp (kUnroll unless given).
template <int U = kUnroll>
__device__ __forceinline__ void score_slice(const float* qs, const uint16_t* __restrict__ Mu, int c0, int c1,
                                            const Arrays& a, int cmax) {
  const int half = (threadIdx.x >> 4) & 1, l16 = threadIdx.x & 15, wid = threadIdx.x >> 5;
  float qv[8];
#pragma unroll
  for (int d = 0; d < 8; ++d) qv[d] = qs[l16 * 8 + d];
  const uint16_t* Ml = Mu + l16 * 8;
  constexpr int kHalfWarps = kThreads / 16;
  // The loop bound is warp-uniform (the shuffles need the whole warp); each
  // half-warp owns chunk base + half + u * kHalfWarps.
  for (int base = c0 + 2 * wid; base < c1; base += kHalfWarps * U) {
    const int cb = base + half;
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = cb + u * kHalfWarps;
      v[u] = (c < c1 && TF_DBG_OK(c >= 0 && c < cmax, kDbgIndexRow)) ? ld_stream16(Ml + (size_t)c * kHeadDim)
                                                                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
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
      if (l16 == 0 && c < c1) {
        const uint32_t key = score_key(s);
        a.keys[c - c0] = key;
        atomicAdd(&a.hist1[key >> 21], 1u);
      }
    }
  }
}

// Round 1 of the cut (requires C > kc; all threads of all CTAs, after
// score_slice and a __syncthreads): the cluster's histogram of the top 11 key
// bits gives the bin b1 holding the kc-th largest key.  Every key with
// (key >> 21) > b1 is selected whatever the rest of the cut.
struct Round1 {
  uint32_t b1;
  int krem1;      // rank of the cut inside bin b1
  int ncand_tot;  // keys of bin b1 over the cluster
};

__device__ __forceinline__ Round1 round1(const Arrays& a, int kc, int S, bool synced = false) {
  __shared__ int s_wsum[kWarps], s_bin, s_krem;
  if (!synced) cluster_sync();  // (synced: a cluster barrier since the histograms were built)
  cluster_sum(a.hist1, a.tot, 2048, S);
  find_bin(a.tot, 2048, kc, s_wsum, &s_bin, &s_krem, CtaBar());
  Round1 r;
  r.b1 = (uint32_t)s_bin;
  r.krem1 = s_krem;
  r.ncand_tot = (int)a.tot[r.b1];
  return r;
}

// Bits 20..0 of the cut from keys gathered on this CTA, a.gcand[0, ng) (keys
// outside bin b1 are skipped; the cut is the krem1-th largest key of the bin),
// then every CTA's counts of keys > T and == T among them (CTA r's keys are
// gcand[roff[r], roff[r + 1])), added to rgt[r] and req[r], and this CTA's
// output offsets.  hist2 and hist3 must be zero.  The group of Bar.
template <class Bar>
__device__ Cut resolve_gathered(const Arrays& a, int ng, uint32_t b1, int krem1, int S, uint32_t rank,
                                const int* roff, int* rgt, int* req, Bar bar) {
  constexpr int NT = Bar::kNT;
  __shared__ int s_wsum[NT / 32], s_bin, s_krem;
  Cut cut;
  cut.b1 = b1;
  cut.cta_eq = 0;
  cut.cta_sel = 0;
  // bits 20..10, then 9..0
  for (int i = threadIdx.x; i < ng; i += NT) {
    const uint32_t key = a.gcand[i];
    if ((key >> 21) == b1) atomicAdd(&a.hist2[(key >> 10) & 2047u], 1u);
  }
  bar();
  find_bin(a.hist2, 2048, krem1, s_wsum, &s_bin, &s_krem, bar);
  const uint32_t pre2 = (b1 << 11) | (uint32_t)s_bin;
  const int krem2 = s_krem;
  for (int i = threadIdx.x; i < ng; i += NT) {
    const uint32_t key = a.gcand[i];
    if ((key >> 10) == pre2) atomicAdd(&a.hist3[key & 1023u], 1u);
  }
  bar();
  find_bin(a.hist3, 1024, krem2, s_wsum, &s_bin, &s_krem, bar);
  cut.T = (pre2 << 10) | (uint32_t)s_bin;
  cut.take_eq = s_krem;
  // per-CTA counts of keys > T and == T among the gathered keys
  for (int i = threadIdx.x; i < ng; i += NT) {
    const uint32_t key = a.gcand[i];
    int r = 0;
    while (r + 1 < S && i >= roff[r + 1]) ++r;
    if (key > cut.T) atomicAdd(&rgt[r], 1);
    if (key == cut.T) atomicAdd(&req[r], 1);
  }
  bar();
  for (int r = 0; r < (int)rank; ++r) {
    cut.cta_sel += rgt[r] + min(max(cut.take_eq - cut.cta_eq, 0), req[r]);
    cut.cta_eq += req[r];
  }
  return cut;
}

// Rest of the cut when the cluster's keys of bin b1 fit the candidate buffer
// (ncand_tot <= cap), run by the group of Bar: each CTA publishes its keys of
// bin b1 and its count of keys above the bin (one cluster barrier, which the
// threads outside the group must also arrive at); every CTA gathers those few
// keys and resolves the remaining 21 bits and every CTA's output offset by
// itself.  hist2 and hist3 must be zero.
template <class Bar>
__device__ Cut fast_cut(const Arrays& a, int n, int S, uint32_t rank, const Round1& r1, Bar bar) {
  constexpr int NT = Bar::kNT;
  __shared__ int s_ncand, s_above, s_roff[kMaxCluster + 1], s_rgt[kMaxCluster], s_req[kMaxCluster];
  const uint32_t b1 = r1.b1;
  const int ncand_tot = r1.ncand_tot;
  if (threadIdx.x == 0) {
    s_ncand = 0;
    s_above = 0;
  }
  bar();
  {
    int above = 0;
    constexpr int k4 = 2048 / NT;
    for (int i = threadIdx.x * k4; i < ((int)threadIdx.x + 1) * k4; ++i) above += (uint32_t)i > b1 ? (int)a.hist1[i] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(&s_above, above);
    for (int i = threadIdx.x; i < n; i += NT) {
      const uint32_t key = a.keys[i];
      if ((key >> 21) == b1) a.cand[atomicAdd(&s_ncand, 1)] = key;  // at most ncand_tot <= cap
    }
  }
  cluster_sync();
  if (threadIdx.x < 32) {
    const int r = threadIdx.x;
    const int nc = r < S ? (int)dsmem_ld_u32(&s_ncand, (uint32_t)r) : 0;
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (r >= o) incl += v;
    }
    if (r < S) {
      s_roff[r] = incl - nc;
      s_rgt[r] = (int)dsmem_ld_u32(&s_above, (uint32_t)r);
      s_req[r] = 0;
    }
    if (r == S - 1) s_roff[S] = incl;
  }
  bar();
  // one remote load per gathered key, all ranks at once; each thread's loads
  // are issued together before any is used
  for (int base = threadIdx.x; base < ncand_tot; base += 4 * NT) {
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * NT;
      int r = 0;
      if (i < ncand_tot)
        while (r + 1 < S && i >= s_roff[r + 1]) ++r;
      v[u] = i < ncand_tot ? dsmem_ld_u32(a.cand + (i - s_roff[r]), (uint32_t)r) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (base + u * NT < ncand_tot) a.gcand[base + u * NT] = v[u];
  }
  bar();
  return resolve_gathered(a, ncand_tot, b1, r1.krem1, S, rank, s_roff, s_rgt, s_req, bar);
}

// Round 1 from a lower bound on the cut (a key that every selected chunk
// reaches, e.g. from the previous decode step's cut): every CTA has listed its
// keys >= the bound in a.cand (*cnt of them; only the first a.cap are stored).
// All threads of all CTAs.  One cluster barrier, then every CTA reads the S
// counts; when the cluster holds between kc and gcap such keys (and no CTA
// more than a.cap), every CTA gathers all of them into a.gcand (room for gcap;
// CTA r's at roff[r] ..) and bin b1 of the kc-th largest key follows from a
// local histogram of those keys (no cluster histogram round; every key of the
// cluster above the bound is gathered, so the cut is the kc-th largest of
// them).  Otherwise (the bound lies above the cut, or admits too many keys)
// nothing that round1 reads has changed, ok is false on every CTA alike, and
// round1 may skip its own cluster barrier.  a.tot is scratch.
struct Hinted {
  bool ok;
  Round1 r1;
  int ntot;  // keys gathered
};

__device__ __forceinline__ Hinted hinted_round1(const Arrays& a, int kc, int S, int gcap, const int* cnt,
                                                int* roff) {
  __shared__ int s_wsum[kWarps], s_bin, s_krem, s_over;
  Hinted h{};
  cluster_sync();
  if (threadIdx.x < 32) {
    const int r = threadIdx.x;
    const int nc = r < S ? (int)dsmem_ld_u32(cnt, (uint32_t)r) : 0;
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (r >= o) incl += v;
    }
    if (r < S) roff[r] = incl - nc;
    if (r == S - 1) roff[S] = incl;
    const unsigned over = __ballot_sync(0xffffffffu, nc > a.cap);
    if (r == 0) s_over = over != 0u;
  }
  for (int i = threadIdx.x; i < 2048; i += kThreads) a.tot[i] = 0;
  __syncthreads();
  const int ntot = roff[S];
  if (ntot < kc || ntot > gcap || s_over) return h;
  for (int base = threadIdx.x; base < ntot; base += 4 * kThreads) {
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * kThreads;
      int r = 0;
      if (i < ntot)
        while (r + 1 < S && i >= roff[r + 1]) ++r;
      v[u] = i < ntot ? dsmem_ld_u32(a.cand + (i - roff[r]), (uint32_t)r) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * kThreads;
      if (i < ntot) {
        a.gcand[i] = v[u];
        atomicAdd(&a.tot[v[u] >> 21], 1u);
      }
    }
  }
  __syncthreads();
  find_bin(a.tot, 2048, kc, s_wsum, &s_bin, &s_krem, CtaBar());
  h.ok = true;
  h.r1.b1 = (uint32_t)s_bin;
  h.r1.krem1 = s_krem;
  h.r1.ncand_tot = (int)a.tot[s_bin];
  h.ntot = ntot;
  return h;
}

// Rest of the cut after hinted_round1 succeeded: the gathered keys hold the
// whole answer, so no cluster barrier.  The group of Bar; hist2 and hist3
// must be zero.
template <class Bar>
__device__ Cut hinted_cut(const Arrays& a, int S, uint32_t rank, const Hinted& h, const int* roff, Bar bar) {
  __shared__ int s_rgt[kMaxCluster], s_req[kMaxCluster];
  if (threadIdx.x < kMaxCluster) {
    s_rgt[threadIdx.x] = 0;
    s_req[threadIdx.x] = 0;
  }
  bar();
  return resolve_gathered(a, h.ntot, h.r1.b1, h.r1.krem1, S, rank, roff, s_rgt, s_req, bar);
}

// Rest of the cut when bin b1 holds more keys than the candidate buffer (huge
// ties or a flat score range): two more cluster-wide histogram rounds resolve
// the last 21 bits, then the CTAs exchange exact counts.  All threads.
static __device__ Cut fallback_cut(const Arrays& a, int n, int S, uint32_t rank, const Round1& r1) {
  __shared__ int s_wsum[kWarps], s_bin, s_krem;
  __shared__ uint32_t s_counts[2];  // keys > T and keys == T in this slice
  const uint32_t b1 = r1.b1;
  Cut cut;
  cut.b1 = b1;
  cut.cta_eq = 0;
  cut.cta_sel = 0;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t key = a.keys[i];
    if ((key >> 21) == b1) atomicAdd(&a.hist2[(key >> 10) & 2047u], 1u);
  }
  cluster_sync();
  cluster_sum(a.hist2, a.tot, 2048, S);
  find_bin(a.tot, 2048, r1.krem1, s_wsum, &s_bin, &s_krem, CtaBar());
  const uint32_t pre2 = (b1 << 11) | (uint32_t)s_bin;
  const int krem2 = s_krem;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t key = a.keys[i];
    if ((key >> 10) == pre2) atomicAdd(&a.hist3[key & 1023u], 1u);
  }
  cluster_sync();
  cluster_sum(a.hist3, a.tot, 1024, S);
  find_bin(a.tot, 1024, krem2, s_wsum, &s_bin, &s_krem, CtaBar());
  cut.T = (pre2 << 10) | (uint32_t)s_bin;
  cut.take_eq = s_krem;
  {
    int ngt = 0, neq = 0;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = a.keys[i];
      ngt += key > cut.T;
      neq += key == cut.T;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ngt += __shfl_xor_sync(0xffffffffu, ngt, o);
      neq += __shfl_xor_sync(0xffffffffu, neq, o);
    }
    if (threadIdx.x == 0) {
      s_counts[0] = 0;
      s_counts[1] = 0;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
      atomicAdd(&s_counts[0], (uint32_t)ngt);
      atomicAdd(&s_counts[1], (uint32_t)neq);
    }
  }
  cluster_sync();
  for (int r = 0; r < (int)rank; ++r) {
    const int gt_r = (int)dsmem_ld_u32(&s_counts[0], (uint32_t)r);
    const int eq_r = (int)dsmem_ld_u32(&s_counts[1], (uint32_t)r);
    cut.cta_sel += gt_r + min(max(cut.take_eq - cut.cta_eq, 0), eq_r);
    cut.cta_eq += eq_r;
  }
  return cut;
}

// Id-order compaction of this CTA's selected chunks by the group of Bar: warp
// w of the group owns local ids [w * seg, (w + 1) * seg).  emit(i, pos, unc)
// is called for every selected local id i with its output position pos (< kc)
// and whether its key lies in bin b1 (a chunk round 1 could not know).
template <class Bar, typename Emit>
__device__ void compact(const Arrays& a, int n, int kc, const Cut& cut, Bar bar, Emit emit) {
  constexpr int NW = Bar::kNT / 32;
  __shared__ int s_wgt[NW], s_weq[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = ((n + NW - 1) / NW + 31) & ~31;
  const int w0 = warp * seg, w1 = min(n, w0 + seg);
  const unsigned lt = (1u << lane) - 1u;
  const uint32_t T = cut.T;
  const int take_eq = cut.take_eq;
  int ngt = 0, neq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? a.keys[i] : 0u;
    ngt += __popc(__ballot_sync(0xffffffffu, i < w1 && key > T));
    neq += __popc(__ballot_sync(0xffffffffu, i < w1 && key == T));
  }
  if (lane == 0) {
    s_wgt[warp] = ngt;
    s_weq[warp] = neq;
  }
  bar();
  int eq_base = cut.cta_eq, sel_base = cut.cta_sel;
  for (int w = 0; w < warp; ++w) {
    sel_base += s_wgt[w] + min(max(take_eq - eq_base, 0), s_weq[w]);
    eq_base += s_weq[w];
  }
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? a.keys[i] : 0u;
    const bool gt = i < w1 && key > T;
    const bool eq = i < w1 && key == T;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_base + __popc(beq & lt) < take_eq);
    const unsigned bsel = __ballot_sync(0xffffffffu, sel);
    const int pos = sel_base + __popc(bsel & lt);
    if (sel && pos < kc) emit(i, pos, (key >> 21) <= cut.b1);
    eq_base += __popc(beq);
    sel_base += __popc(bsel);
  }
}

}  // namespace topk
}  // namespace tf
