// a2 + a3 + a4 (+ a5) fused -- the Force 2 retrieval drafter's decode attention
// in one launch: chunk scores, top-k selection and attention over the selected
// chunks; optionally (a6) the Force 1 drafter's sink + window attention of the
// same queries in the same launch.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": the retrieval drafter is the target model attending only to the
// KV blocks whose key-query similarity is highest, within a fixed budget.
// Outputs are those of the top-k call (idx, n_sel, s_cut) and of the sparse
// attention call over that selection (out), computed in one pass.
//
// Design: the top-k cluster (one cluster of S <= 16 CTAs per (b, g) unit, CTA r
// scoring the r-th slice of the chunk means; see topk_select.cuh) keeps going
// after the cut: each CTA attends the chunks it selected itself, so no chunk
// list goes through global memory and no second launch waits for the first.
//  * After the first cluster histogram round fixes the bin b1 of the cut,
//    every chunk whose key lies above b1 is selected whatever the rest of the
//    cut.  The CTA lists those chunks and splits: warps 0..7 finish the cut
//    (candidate gather, last 21 bits, id-order output, the chunks of bin b1
//    appended to the list) on a named barrier, while warps 8..15 attend the
//    listed chunks.  When the cut is done, warps 0..7 join them.  HBM keeps
//    streaming while the cut is resolved.
//  * Each warp owns one 4 KB ring slot and stages its own chunks: lane 0
//    claims the next list entry (a shared counter), copies the chunk's K and V
//    rows into the slot (one query head: cp.async.bulk; two to four: two TMA
//    boxes in the 128-byte swizzle) and the warp waits for them; entries past
//    the certain ones are read once the cut group has published the final
//    list.  No hand-over between warps: a slot is free again as soon as its
//    warp has read it.
//  * One query head: consumer lane (row r, quarter dq) forms 32-dim dot
//    products with the query row held in shared memory in a bank-conflict-free
//    permuted layout, and owns 4 head dims of P V.  Two to four heads: the
//    warp runs Q K^T and P V on the tensor cores (mma.sync fragments).  The
//    online softmax runs in the log2 domain in fp32.
//  * The window form (template WIN, two to four heads): the sink and window
//    keys join the certain entries as pieces of up to 8 rows, and the MMA
//    tile's B-fragment rows 4..7, idle with at most four heads, carry the same
//    queries masked to those pieces; rows 0..3 are masked to the retrieved
//    chunks.  The merges carry all 8 rows; rows 4.. go to the window output.
//  * Warps merge in shared memory, then CTA rank 0 merges the S partial states
//    of the cluster through distributed shared memory (log-sum-exp identity)
//    and writes the output; both merges compute each (warp or rank, row)
//    scale once and then sum float4s.
// All waits are bounded; a timeout (only a hardware fault can cause one)
// leaves NaN in the outputs.
#include <cuda_bf16.h>

#include "tma_host.cuh"
#include "topk_select.cuh"

namespace tf {
namespace {

using namespace sm100;
using topk::kMaxCluster;
using topk::kMaxSliceKeys;
using topk::kThreads;
using topk::kWarps;

constexpr int kComputeWarps = kWarps;                   // every warp attends
constexpr int kCutWarps = 8;                            // warps 0..7 finish the cut
constexpr int kRingSlots = kComputeWarps;               // one slot per warp
constexpr int kEarlySlots = kComputeWarps - kCutWarps;  // slots of warps 8..15
// A ring slot holds one chunk's 8 K rows at [0, 2 KB) and its 8 V rows at
// [2 KB, 4 KB).  One query head: rows 256 bytes apart (one bulk copy each).
// Two to four heads (tensor-core consumers): each 2 KB piece is two 1 KB
// swizzle atoms (dims 0..63, 64..127; 16-byte unit u of row r at
// r * 128 + ((u ^ r) * 16)), written by one TMA box, so that the eight rows an
// ldmatrix reads fall in distinct banks.
constexpr int kSlotBytes = 4096;
constexpr int kQPitch = 272;  // bytes between the bf16 query rows (conflict-free ldmatrix)
constexpr int kCandCap = 2048;    // keys of the threshold bin gathered on every CTA
constexpr int kHintCap = 4096;    // keys above a cut bound gathered on every CTA (over gcand and hist1)
constexpr int kMaxList = 2048;    // selected chunks per CTA (kc <= kMaxList)
constexpr uint32_t kIdleLimit = 1u << 22;  // polls for the final list before a warp gives up

// Dynamic shared memory (bytes).
// (from a 1 KB-aligned base, so that every slot starts a swizzle atom)
//  [0, 32768)      ring slots 0..7 (warps 8..15); during round 1 they hold
//                  tot, which only this CTA reads
//  [32768, 65536)  ring slots 8..15 (warps 0..7) once the cut is done;
//                  until then hist2, hist3, gcand (the cut group's scratch)
//                  and hist1 (read by the other CTAs in round 1, which they
//                  finish before the cut's cluster barrier; with a cut bound
//                  that holds, no round 1 runs and gcand extends over it)
//  cand            read by the other CTAs until the end of their cut: never overlaid
//  alist           this CTA's selected chunks (certain ones first)
//  keys            this CTA's score keys
constexpr int kOffTot = 0;
constexpr int kOffHist2 = kEarlySlots * kSlotBytes;  // 32768
constexpr int kOffHist3 = kOffHist2 + 2048 * 4;      // 40960
constexpr int kOffGcand = kOffHist3 + 1024 * 4;      // 45056
constexpr int kOffHist1 = kOffGcand + kCandCap * 4;  // 53248
constexpr int kOffCand = kRingSlots * kSlotBytes;    // 65536
constexpr int kOffList = kOffCand + kCandCap * 4;    // 73728
constexpr int kOffKeys = kOffList + kMaxList * 4;    // 81920
static_assert(kOffHist1 + 2048 * 4 <= kOffCand, "the cut's scratch must fit the late slots");
static_assert(kOffGcand + kHintCap * 4 <= kOffCand, "the hinted gather must fit the late slots");
static_assert(kOffTot + 2048 * 4 <= kOffHist2, "tot must stay inside the early slots");

struct DraftParams {
  const uint16_t* q;  // [B, Hq, 128]
  const uint16_t* M;  // [B, Hkv, Cmax, 128]
  const uint16_t* K;  // [B, Hkv, Lmax, 128]
  const uint16_t* V;
  const int32_t* seq_lens;
  int Hq, Hkv, Lmax, kc;
  float scale_log2;  // softmax scale * log2(e)
  int32_t* idx;      // [B, Hkv, kc]
  int32_t* n_sel;    // [B, Hkv]
  float* s_cut;      // [B, Hkv] or null
  float* out;        // [B, Hq, 128]
  const float* hint;  // [B, Hkv] lower bounds on the cut scores, or null (NaN: none for that unit)
  int nseq;           // B
  int longest_first;  // 1: block row r serves the sequence with the r-th longest context (B <= 64)
  CUtensorMap mapK, mapV;  // two to four heads: 8-row pieces of K and V as [B * Hkv * Lmax, 128] boxes
  // optional, two to four heads: the sink + window attention of the same
  // queries, written to wout [B, Hq, 128] (null: none)
  float* wout;
  int n_sink, window;
};

// + 1 KB to align the base
size_t draft_smem(int slice) { return 1024 + (size_t)kOffKeys + (size_t)slice * sizeof(uint32_t); }

// Warp-level tensor-core fragments (mma.sync: a chunk of 8 keys is far below
// the 64-row minimum of a tcgen05 tile).  ldsm_x4 / ldsm_x4_t: four 8 x 8
// 16-bit matrices from shared memory, lane i giving the address of row i % 8
// of matrix i / 8 (_t: transposed).  mma_s: C += A B for a 16 x 16 A whose
// rows 8..15 are zero (a0: rows 0..7, k 0..7; a2: k 8..15), B 16 x 8.
// mma_pv: C += A B for A 16 x 8, B 8 x 8.  bf16 operands, fp32 accumulators.
__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
  uint32_t u;
  memcpy(&u, &v, sizeof(u));
  return u;
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_s(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
               "{%8, %9}, {%0, %1, %2, %3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_pv(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
               "{%0, %1, %2, %3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a0), "r"(a1), "r"(b0));
}

// Ring slot of warp w: warps 8..15 take slots 0..7, warps 0..7 (the cut
// group) slots 8..15.
__device__ __forceinline__ int slot_of(int warp) { return (warp + kEarlySlots) % kRingSlots; }

template <int NQ, bool WIN>
__global__ void __launch_bounds__(kThreads, 2) retrieval_draft_kernel(const __grid_constant__ DraftParams p) {
  static_assert(!WIN || NQ >= 2, "the window rows ride in the tensor-core consumers' fragments");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* const smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(16) float qsm[NQ * kHeadDim];  // scaled query rows, permuted (see below)
  __shared__ float qs[kHeadDim];                      // the group's summed query (scores)
  // two to four heads: the query rows as bf16, 8 rows (heads past G zero) 272 bytes apart
  __shared__ __align__(16) uint16_t qbf[NQ >= 2 ? kChunk * kQPitch / 2 : 8];
  __shared__ __align__(8) uint64_t bar_full[kRingSlots];
  __shared__ int slot_n[kRingSlots], slot_uses[kRingSlots];
  // rows of a warp's state: the heads (NQ), or with a window output all 8
  // fragment rows: heads 0..3, then the window rows 4..7
  constexpr int kRowsW = WIN ? 8 : NQ;
  __shared__ float wm[kComputeWarps][kRowsW], wl[kComputeWarps][kRowsW];
  __shared__ __align__(16) float cpart[kRowsW][kHeadDim];
  __shared__ float cm[kRowsW], cl[kRowsW];
  __shared__ uint8_t slot_win[kRingSlots];  // 1: the slot holds a window piece
  __shared__ uint32_t s_min;
  __shared__ int s_na, s_ntot, s_abort, s_hcnt, s_next;
  __shared__ int s_wg[4];  // window geometry: sinks kept, first window key, sink pieces, pieces
  __shared__ int s_hroff[kMaxCluster + 1];
  __shared__ volatile int s_cut_done;

  uint8_t* ring = smem;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kOffKeys);
  int32_t* alist = reinterpret_cast<int32_t*>(smem + kOffList);
  const topk::Arrays a{keys,
                       reinterpret_cast<uint32_t*>(smem + kOffHist1),
                       reinterpret_cast<uint32_t*>(smem + kOffHist2),
                       reinterpret_cast<uint32_t*>(smem + kOffHist3),
                       reinterpret_cast<uint32_t*>(smem + kOffTot),
                       reinterpret_cast<uint32_t*>(smem + kOffCand),
                       reinterpret_cast<uint32_t*>(smem + kOffGcand),
                       kCandCap};

  const int S = (int)gridDim.x;  // the cluster spans grid x
  const uint32_t rank = cluster_ctarank();
  const int g = (int)blockIdx.y % p.Hkv;
  const int G = p.Hq / p.Hkv;  // <= NQ
  const int Cmax = (p.Lmax + kChunk - 1) / kChunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingSlots; ++s) mbar_init(&bar_full[s], 1);
    s_abort = 0;
    s_next = 0;
    s_hcnt = 0;
    s_na = 0;
    s_cut_done = 0;
    s_min = 0xffffffffu;
    fence_mbar_init();
  }
  topk::zero_hists(a);
  pdl_wait();
  // Ragged batches: clusters start in about block order, so block row r takes
  // the sequence with the r-th longest context (ties in batch order; every
  // warp ranks the at most 64 lengths with shuffles and one ballot) and the
  // longest units do not start in the last wave.
  int b = (int)blockIdx.y / p.Hkv;
  if (p.longest_first) {
    const int slot = b;
    const int l0 = lane < p.nseq ? clamp_len(p.seq_lens[lane], p.Lmax) : -1;
    const int l1 = lane + 32 < p.nseq ? clamp_len(p.seq_lens[lane + 32], p.Lmax) : -1;
    int r0 = 0, r1 = 0;
    for (int j = 0; j < p.nseq; ++j) {
      const int lj = __shfl_sync(0xffffffffu, j < 32 ? l0 : l1, j & 31);
      r0 += (lj > l0 || (lj == l0 && j < lane)) ? 1 : 0;
      r1 += (lj > l1 || (lj == l1 && j < lane + 32)) ? 1 : 0;
    }
    const unsigned m0 = __ballot_sync(0xffffffffu, lane < p.nseq && r0 == slot);
    const unsigned m1 = __ballot_sync(0xffffffffu, lane + 32 < p.nseq && r1 == slot);
    b = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
  }
  const int unit = b * p.Hkv + g;
  const int L = clamp_len(p.seq_lens[b], p.Lmax);
  const int C = (L + kChunk - 1) / kChunk;
  const int per = (C + S - 1) / S;
  const int c0 = min(C, (int)rank * per);
  const int c1 = min(C, c0 + per);
  const int n = c1 - c0;

  // Queries.  Head h's scaled row is stored so that the 16-byte piece of dims
  // [32 dq + 8 jr + 4 hf, +4) sits at 16-byte unit hf * 16 + 4 dq + jr: the
  // eight (dq, jr) pairs read together by a quarter-warp below then fall in
  // eight different bank groups.
  const uint16_t* qg = p.q + ((size_t)b * p.Hq + (size_t)g * G) * kHeadDim;
  if (threadIdx.x < kHeadDim) {
    float s = 0.0f;
    for (int h = 0; h < G; ++h) s += __uint_as_float((uint32_t)qg[h * kHeadDim + threadIdx.x] << 16);
    qs[threadIdx.x] = s;
  }
  for (int e = threadIdx.x; e < NQ * kHeadDim; e += kThreads) {
    const int h = e / kHeadDim, d = e % kHeadDim;
    const float v = h < G ? __uint_as_float((uint32_t)qg[h * kHeadDim + d] << 16) * p.scale_log2 : 0.0f;
    const int u = ((d >> 2) & 1) * 16 + 4 * (d >> 5) + ((d >> 3) & 3);
    qsm[h * kHeadDim + u * 4 + (d & 3)] = v;
  }
  if constexpr (NQ >= 2) {
    for (int e = threadIdx.x; e < kChunk * kQPitch / 2; e += kThreads) {
      const int h = e / (kQPitch / 2), d = e % (kQPitch / 2);
      // rows 0..G-1 the heads; with a window output rows 4..4+G-1 the same heads again
      const int hq = h < G ? h : ((WIN && h >= 4 && h - 4 < G) ? h - 4 : -1);
      qbf[e] = (hq >= 0 && d < kHeadDim) ? qg[hq * kHeadDim + d] : (uint16_t)0;
    }
  }
  __syncthreads();
  topk::score_slice<8>(qs, p.M + (size_t)unit * Cmax * kHeadDim, c0, c1, a, Cmax);
  __syncthreads();

  const uint16_t* Ku = p.K + (size_t)unit * p.Lmax * kHeadDim;
  const uint16_t* Vu = p.V + (size_t)unit * p.Lmax * kHeadDim;
  // window pieces of this unit (with a window output): the sinks
  // [0, ns_eff) and the recent keys [w0, L) in pieces of up to 8 rows; list
  // entry -1 - k is piece k.  Lane 0 reads the geometry from shared memory
  // when it stages a window piece.
  constexpr bool win = WIN;
  int n_pw = 0;
  if (win) {
    const int ns_eff = min(p.n_sink, L), w0 = max(p.n_sink, L - p.window);
    const int n_sp = (ns_eff + kChunk - 1) / kChunk;
    n_pw = n_sp + (max(L - w0, 0) + kChunk - 1) / kChunk;
    if (threadIdx.x == 0) {
      s_wg[0] = ns_eff;
      s_wg[1] = w0;
      s_wg[2] = n_sp;
      s_wg[3] = n_pw;
    }
  }
  auto piece = [&](int k, int& y, int& nr) {
    if (k < s_wg[2]) {
      y = k * kChunk;
      nr = min(kChunk, s_wg[0] - y);
    } else {
      y = s_wg[1] + (k - s_wg[2]) * kChunk;
      nr = min(kChunk, L - y);
    }
  };

  // Stage chunk c (its valid rows of K and of V) into a ring slot.  An id
  // outside [0, C) cannot come out of the selection; it is refused all the
  // same (the slot completes empty and the outputs are poisoned) rather than
  // turned into a copy from outside the cache.
  auto issue = [&](int slot, int c) {
    if (c < 0 || c >= C) {
      atomicExch(&s_abort, 1);
      slot_n[slot] = 0;
      mbar_arrive(&bar_full[slot]);
      return;
    }
    const int y = c * kChunk;
    int nr = min(kChunk, L - y);
    if (!TF_DBG_OK(nr > 0 && y + nr <= L && L <= p.Lmax, kDbgCacheRow)) nr = 0;
    slot_n[slot] = nr;
    const uint32_t bytes = (uint32_t)nr * kHeadDim * 2;
    uint8_t* dst = ring + slot * kSlotBytes;
    mbar_arrive_expect_tx(&bar_full[slot], 2 * bytes);
    bulk_load(dst, Ku + (size_t)y * kHeadDim, bytes, &bar_full[slot]);
    bulk_load(dst + 2048, Vu + (size_t)y * kHeadDim, bytes, &bar_full[slot]);
  };
  // The same for the tensor-core consumers (lane 0): one TMA box for the K
  // piece and one for the V piece, always 8 rows (rows past the context hold
  // whatever the cache holds there, zero past its end; they are masked below)
  auto issue_tma = [&](int slot, int c) {
    // a chunk id, or -1 - k for window piece k
    int y = 0, nr = 0;
    bool ok = c >= 0 && c < C;
    if constexpr (WIN) ok = c >= 0 ? c < C : (-1 - c) < s_wg[3];
    if (ok) {
      if (c >= 0) {
        y = c * kChunk;
        nr = min(kChunk, L - y);
      } else {
        piece(-1 - c, y, nr);
      }
    }
    if (ok && !TF_DBG_OK(nr > 0 && y >= 0 && y + nr <= L && L <= p.Lmax, kDbgCacheRow)) nr = 0;
    if (!ok) atomicExch(&s_abort, 1);
    slot_n[slot] = nr;
    if constexpr (WIN) slot_win[slot] = c < 0 ? 1 : 0;
    if (nr == 0) {
      mbar_arrive(&bar_full[slot]);
      return;
    }
    uint8_t* dst = ring + slot * kSlotBytes;
    const int row = (int)((size_t)unit * p.Lmax + y);
    mbar_arrive_expect_tx(&bar_full[slot], (uint32_t)kSlotBytes);
    tma_load_3d(dst, &p.mapK, &bar_full[slot], 0, row, 0);
    tma_load_3d(dst + 2048, &p.mapV, &bar_full[slot], 0, row, 0);
  };

  int32_t* out_idx = p.idx + (size_t)unit * p.kc;
  uint32_t T = 0;
  bool split = false;  // warps 0..7 finish the cut while the others attend
  topk::Round1 r1{};
  topk::Hinted hinted{};
  if (C <= p.kc) {
    // Every chunk is selected: ids in order, slots past C hold -1, s_cut = min score.
    uint32_t mn = 0xffffffffu;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      out_idx[c0 + i] = c0 + i;
      alist[i] = c0 + i;
      mn = min(mn, keys[i]);
    }
    if (rank == 0)
      for (int i = C + (int)threadIdx.x; i < p.kc; i += kThreads) out_idx[i] = -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    if (lane == 0) atomicMin(&s_min, mn);
    if (threadIdx.x == 0) {
      s_na = n;
      s_ntot = n;
    }
  } else {
    // With a lower bound on the cut, list the keys that reach it; if the
    // cluster holds between kc and kHintCap of them, the cut comes from those
    // keys alone (one cluster barrier, no cluster histogram round, no second
    // barrier for the rest of the cut).  Otherwise the unhinted path runs,
    // with the barrier already passed; the selection is the same either way.
    const float hv = p.hint ? p.hint[unit] : NAN;
    if (hv == hv) {
      const uint32_t hkey = score_key(hv);
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t key = keys[i];
        if (key >= hkey) {
          const int at = atomicAdd(&s_hcnt, 1);
          if (at < kCandCap) a.cand[at] = key;
        }
      }
      __syncthreads();
      hinted = topk::hinted_round1(a, p.kc, S, kHintCap, &s_hcnt, s_hroff);
    }
    // after a bound that did not hold, round 1 needs no barrier of its own
    r1 = hinted.ok ? hinted.r1 : topk::round1(a, p.kc, S, hv == hv);
    // chunks above bin b1: selected whatever the rest of the cut (list order is free)
    for (int i = threadIdx.x; i < n; i += kThreads)
      if ((keys[i] >> 21) > r1.b1) alist[atomicAdd(&s_na, 1)] = c0 + i;
    __syncthreads();
    if (threadIdx.x == 0) s_ntot = s_na;
    split = hinted.ok || r1.ncand_tot <= kCandCap;
    if (!split) {
      // rare: resolve the cut with every warp, attend afterwards
      __syncthreads();
      const topk::Cut cut = topk::fallback_cut(a, n, S, rank, r1);
      T = cut.T;
      topk::compact(a, n, p.kc, cut, topk::CtaBar(), [&](int i, int pos, bool unc) {
        out_idx[pos] = c0 + i;
        if (unc) {
          const int at = atomicAdd(&s_ntot, 1);
          if (at < kMaxList) alist[at] = c0 + i;
        }
      });
    }
  }
  if (win) {
    // this CTA's window pieces (k = rank, rank + S, ...), known before the cut:
    // appended to the certain entries while the cut runs (split), else to
    // the final list
    __syncthreads();
    const int base = split ? s_na : s_ntot;
    const int mine = n_pw > (int)rank ? (n_pw - (int)rank + S - 1) / S : 0;
    if (base + mine > kMaxList) {
      if (threadIdx.x == 0) atomicExch(&s_abort, 1);  // cannot happen within the host's limits
    } else {
      for (int j = threadIdx.x; j < mine; j += kThreads) alist[base + j] = -1 - ((int)rank + j * S);
    }
    __syncthreads();
    if (threadIdx.x == 0 && base + mine <= kMaxList) {
      if (split) s_na = base + mine;
      s_ntot = base + mine;
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- attention
  const int rows = G < NQ ? G : NQ;
  float m[NQ], l[NQ], o[NQ][4];
  // two to four heads (tensor-core consumers): lane (g, t) = (lane / 4, lane % 4)
  // keeps the running max and sum of fragment row g (head g; in the window
  // form rows 4..7 are the window rows), and oc[bk] the output of dims
  // 16 bk + g and 16 bk + g + 8 for rows 2t and 2t + 1
  float mh = -INFINITY, lh = 0.0f;
  float oc[NQ >= 2 ? 8 : 1][4];
#pragma unroll
  for (int bk = 0; bk < (NQ >= 2 ? 8 : 1); ++bk)
#pragma unroll
    for (int i = 0; i < 4; ++i) oc[bk][i] = 0.0f;
#pragma unroll
  for (int h = 0; h < NQ; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[h][i] = 0.0f;
  }
  const bool cut_group = split && warp < kCutWarps;
  if (cut_group) {
    // ---- warps 0..7: the rest of the cut, then attention from slots 8..15
    const topk::Cut cut = hinted.ok ? topk::hinted_cut(a, S, rank, hinted, s_hroff, topk::Warps0to7Bar())
                                    : topk::fast_cut(a, n, S, rank, r1, topk::Warps0to7Bar());
    T = cut.T;
    topk::compact(a, n, p.kc, cut, topk::Warps0to7Bar(), [&](int i, int pos, bool unc) {
      out_idx[pos] = c0 + i;
      if (unc) {
        const int at = atomicAdd(&s_ntot, 1);
        if (at < kMaxList) alist[at] = c0 + i;
      }
    });
    topk::Warps0to7Bar()();
    if (threadIdx.x == 0) {
      __threadfence_block();
      s_cut_done = 1;
    }
  } else if (split && !hinted.ok) {
    cluster_arrive();  // the cut group's one cluster barrier; waited for below
  }

  {
    // ---------------------------------------------------------------- attention
    // Lane 0 claims the next list entry and stages the chunk into the warp's
    // slot.  Entries [0, ncert) are final when the attention starts; with the
    // cut still running, later entries are read once the cut group has
    // published the final length.
    const int slot = slot_of(warp);
    const int ncert = split ? s_na : min(s_ntot, kMaxList);
    // lane = (row r, quarter dq); pieces visited in the rotated order jr(j)
    const int r = lane >> 2, dq = lane & 3;
    const int rot = (dq >> 1) + 2 * (r & 1);
    const float4* q4 = reinterpret_cast<const float4*>(qsm);
    const uint8_t* kb = ring + slot * kSlotBytes;
    const uint8_t* vb = kb + 2048;
    constexpr int kNoChunk = -0x7fffffff - 1;
    uint32_t u = 0;  // copies issued into the slot
    while (true) {
      int c = kNoChunk;
      if (lane == 0) {
        const int i = atomicAdd(&s_next, 1);
        if (i < ncert) {
          c = alist[i];
        } else if (split) {
          uint32_t spins = 0;
          while (!s_cut_done && !*(volatile int*)&s_abort) {
            if (++spins > kIdleLimit) {
              atomicExch(&s_abort, 1);
              break;
            }
            __nanosleep(64);
          }
          if (s_cut_done) {
            __threadfence_block();
            if (i < min(*(volatile int*)&s_ntot, kMaxList)) c = alist[i];
          }
        }
        if (c != kNoChunk) {
          fence_proxy_async_smem();  // the slot's earlier generic reads and writes before the copy
          if constexpr (NQ == 1) issue(slot, c);
          else issue_tma(slot, c);
        }
      }
      c = __shfl_sync(0xffffffffu, c, 0);
      if (c == kNoChunk) break;
      const uint32_t ph = u & 1;
      ++u;
      if (!mbar_wait(&bar_full[slot], ph)) {
        if (lane == 0) atomicExch(&s_abort, 1);
        break;
      }
      const int nr = slot_n[slot];
      if constexpr (NQ == 1) {
        float sa[NQ], sb[NQ];  // two independent partial sums per head
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int jr = (j + rot) & 3;
          const uint4 kv = *reinterpret_cast<const uint4*>(kb + r * 256 + dq * 64 + jr * 16);
          float f[8];
          unpack8(kv, f);
#pragma unroll
          for (int h = 0; h < NQ; ++h) {
            const float4 qa = q4[h * 32 + 4 * dq + jr];
            const float4 qb = q4[h * 32 + 16 + 4 * dq + jr];
            float t = qa.x * f[0];
            t = fmaf(qa.y, f[1], t);
            t = fmaf(qa.z, f[2], t);
            t = fmaf(qa.w, f[3], t);
            t = fmaf(qb.x, f[4], t);
            t = fmaf(qb.y, f[5], t);
            t = fmaf(qb.z, f[6], t);
            t = fmaf(qb.w, f[7], t);
            if (j == 0) sa[h] = t;
            else if (j == 1) sb[h] = t;
            else if (j == 2) sa[h] += t;
            else sb[h] += t;
          }
        }
        const bool valid = r < nr;
        float pr[NQ];
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          float s = sa[h] + sb[h];
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          s += __shfl_xor_sync(0xffffffffu, s, 2);
          s = valid ? s : -INFINITY;
          float cmx = s;
          cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 4));
          cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 8));
          cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 16));
          const float mn = fmaxf(m[h], cmx);
          const float alpha = merge_scale(m[h], mn);
          pr[h] = (s == -INFINITY) ? 0.0f : exp2f(s - mn);
          float ps = pr[h];
          ps += __shfl_xor_sync(0xffffffffu, ps, 4);
          ps += __shfl_xor_sync(0xffffffffu, ps, 8);
          ps += __shfl_xor_sync(0xffffffffu, ps, 16);
          l[h] = l[h] * alpha + ps;
          m[h] = mn;
#pragma unroll
          for (int i = 0; i < 4; ++i) o[h][i] *= alpha;
        }
        // P V: lane owns head dims [4 lane, 4 lane + 4) of every row
        for (int rr = 0; rr < nr; ++rr) {
          const uint2 vv = *reinterpret_cast<const uint2*>(vb + rr * 256 + lane * 8);
          const float v0 = __uint_as_float(vv.x << 16), v1 = __uint_as_float(vv.x & 0xffff0000u);
          const float v2 = __uint_as_float(vv.y << 16), v3 = __uint_as_float(vv.y & 0xffff0000u);
#pragma unroll
          for (int h = 0; h < NQ; ++h) {
            const float pw = __shfl_sync(0xffffffffu, pr[h], rr * 4);  // lane 4 rr holds row rr
            o[h][0] = fmaf(pw, v0, o[h][0]);
            o[h][1] = fmaf(pw, v1, o[h][1]);
            o[h][2] = fmaf(pw, v2, o[h][2]);
            o[h][3] = fmaf(pw, v3, o[h][3]);
          }
        }
      } else if (nr > 0) {
        // S[h][key] = q_h . K_key on the tensor cores (heads as rows, zero past
        // G), then the online softmax per head and O^T += V^T P^T with P split
        // into bf16 hi and lo parts (P to 2^-17, as the verify kernel does)
        const int t4 = lane & 3;
        const uint32_t kaddr = smem_u32(ring + slot * kSlotBytes);
        const uint32_t vaddr = kaddr + 2048;
        const uint32_t qaddr = smem_u32(qbf);
        if (nr < kChunk) {
          // rows past the chunk's end may hold anything: zero them in V so
          // that 0 * V stays 0 (their scores are masked below)
          uint8_t* vp = ring + slot * kSlotBytes + 2048;
          for (int e = lane; e < (kChunk - nr) * 16; e += 32)
            *reinterpret_cast<uint4*>(vp + ((e >> 3) & 1) * 1024 + (nr + (e >> 4)) * 128 + (e & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          __syncwarp();
        }
        // ldmatrix row addresses: lane = (matrix m = lane / 8, row r = lane % 8);
        // 16-byte unit u of a piece row sits in atom u / 8 at ((u % 8) ^ r) * 16
        const int lr = lane & 7, lm = lane >> 3;
        auto piece_addr = [&](uint32_t base, int u) -> uint32_t {
          return base + (uint32_t)((u >> 3) * 1024 + lr * 128 + (((u & 7) ^ lr) << 4));
        };
        const uint32_t q_off = (uint32_t)(lr * kQPitch + lm * 16);
        float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ks += 2) {  // 32 dims per step
          uint32_t qa[4], kf[4];
          ldsm_x4(qa, qaddr + q_off + ks * 32);
          ldsm_x4(kf, piece_addr(kaddr, 2 * ks + lm));
          mma_s(sc, qa[0], qa[1], kf[0], kf[1]);
          mma_s(sc, qa[2], qa[3], kf[2], kf[3]);
        }
        // this lane: row g8 (heads 0..3, window rows 4..7), keys 2 t4 and 2 t4 + 1;
        // a chunk feeds the head rows, a window piece the window rows
        bool row_on = true;  // without a window output rows past G hold zero queries, discarded
        if constexpr (WIN) row_on = slot_win[slot] ? (lane >> 2) >= 4 : (lane >> 2) < 4;
        const float s0 = (row_on && 2 * t4 < nr) ? sc[0] * p.scale_log2 : -INFINITY;
        const float s1 = (row_on && 2 * t4 + 1 < nr) ? sc[1] * p.scale_log2 : -INFINITY;
        float cmx = fmaxf(s0, s1);
        cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 1));
        cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 2));
        const float mn = fmaxf(mh, cmx);
        const float alpha = merge_scale(mh, mn);
        const float p0 = (s0 == -INFINITY) ? 0.0f : exp2f(s0 - mn);
        const float p1 = (s1 == -INFINITY) ? 0.0f : exp2f(s1 - mn);
        float ps = p0 + p1;
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        lh = lh * alpha + ps;
        mh = mn;
        // this lane's outputs belong to heads 2 t4 and 2 t4 + 1
        const float ae = __shfl_sync(0xffffffffu, alpha, 8 * t4);
        const float ao = __shfl_sync(0xffffffffu, alpha, 8 * t4 + 4);
        const __nv_bfloat162 ph2 = __floats2bfloat162_rn(p0, p1);
        const __nv_bfloat162 pl2 = __floats2bfloat162_rn(p0 - __low2float(ph2), p1 - __high2float(ph2));
        const uint32_t bh = bf16x2_bits(ph2), bl = bf16x2_bits(pl2);
#pragma unroll
        for (int bk = 0; bk < 8; bk += 2) {  // 32 dims per step
          uint32_t va[4];
          ldsm_x4_t(va, piece_addr(vaddr, 2 * bk + lm));
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            float (&cc)[4] = oc[bk + hb];
            cc[0] *= ae;
            cc[1] *= ao;
            cc[2] *= ae;
            cc[3] *= ao;
            mma_pv(cc, va[2 * hb], va[2 * hb + 1], bh);
            mma_pv(cc, va[2 * hb], va[2 * hb + 1], bl);
          }
        }
      }
      __syncwarp();
    }
    if (lane == 0) slot_uses[slot] = (int)u;
  }
  if (split && !cut_group && !hinted.ok) cluster_wait();
  __syncthreads();  // every chunk consumed: the ring is idle and serves as scratch
  if (s_abort && threadIdx.x == 0) {
    // (only after a timeout) let every copy still in flight land before the
    // ring is reused or the CTA exits
    for (int sl = 0; sl < kRingSlots; ++sl)
      if (slot_uses[sl] > 0) mbar_wait(&bar_full[sl], (slot_uses[sl] - 1) & 1, 1u << 8);
  }
  __syncthreads();
  // Each warp's state: wo [kComputeWarps][kRowsW][128] over the idle ring.
  // The tensor-core consumers' fragment rows 2 t4 and 2 t4 + 1 store with the
  // column XOR-ed by 8 t4 (the four lanes of a quarter then write four bank
  // groups); groups of four columns stay contiguous, so reads take float4s.
  float* wo = reinterpret_cast<float*>(ring);
  auto wo_col = [](int h, int d) { return NQ >= 2 ? d ^ (((h >> 1) & 3) << 3) : d; };
  const int nrows = win ? 2 * rows : rows;  // merged rows: the heads, then the window rows
  auto row_of = [&](int i) { return i < rows ? i : 4 + (i - rows); };
  if constexpr (NQ == 1) {
    if (lane == 0) {
      wm[warp][0] = m[0];
      wl[warp][0] = l[0];
    }
    *reinterpret_cast<float4*>(wo + warp * kRowsW * kHeadDim + lane * 4) = make_float4(o[0][0], o[0][1], o[0][2], o[0][3]);
  } else {
    const int g8 = lane >> 2, t4 = lane & 3;
    if (t4 == 0 && g8 < kRowsW) {
      wm[warp][g8] = mh;
      wl[warp][g8] = lh;
    }
    if (2 * t4 < kRowsW) {  // rows 2 t4 and 2 t4 + 1
#pragma unroll
      for (int bk = 0; bk < 8; ++bk)
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int h = 2 * t4 + hb;
          float* row = wo + (warp * kRowsW + h) * kHeadDim;
          row[wo_col(h, 16 * bk + g8)] = oc[bk][hb];
          row[wo_col(h, 16 * bk + g8 + 8)] = oc[bk][2 + hb];
        }
    }
  }
  __syncthreads();

  // ---- this CTA's partial state: merge the compute warps.  The scale of
  // (warp, row) is computed once; the outputs are float4 weighted sums.
  __shared__ float wf[kComputeWarps][kRowsW];
  if (threadIdx.x < nrows) {
    const int h = row_of(threadIdx.x);
    float mx = -INFINITY;
    for (int w = 0; w < kComputeWarps; ++w) mx = fmaxf(mx, wm[w][h]);
    cm[h] = mx;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kComputeWarps * nrows; e += kThreads) {
    const int w = e / nrows, h = row_of(e % nrows);
    wf[w][h] = merge_scale(wm[w][h], cm[h]);
  }
  __syncthreads();
  if (threadIdx.x < nrows) {
    const int h = row_of(threadIdx.x);
    float ls = 0.0f;
    for (int w = 0; w < kComputeWarps; ++w) ls = fmaf(wf[w][h], wl[w][h], ls);
    cl[h] = ls;
  }
  for (int e = threadIdx.x; e < nrows * (kHeadDim / 4); e += kThreads) {
    const int h = row_of(e / (kHeadDim / 4)), d = 4 * (e % (kHeadDim / 4));
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int w = 0; w < kComputeWarps; ++w) {
      const float f = wf[w][h];
      const float4 v = *reinterpret_cast<const float4*>(wo + (w * kRowsW + h) * kHeadDim + wo_col(h, d));
      acc.x = fmaf(f, v.x, acc.x);
      acc.y = fmaf(f, v.y, acc.y);
      acc.z = fmaf(f, v.z, acc.z);
      acc.w = fmaf(f, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(&cpart[h][d]) = acc;
  }
  cluster_sync();

  // ---- rank 0 merges the cluster's partial states and writes the outputs:
  // the scale of (rank, row), divided by the row's total, once; then 16-byte
  // loads of every rank's partial outputs
  if (rank == 0) {
    __shared__ float rf[kMaxCluster][kRowsW];
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    for (int e = threadIdx.x; e < S * nrows; e += kThreads) {
      const int rr = e / nrows, h = row_of(e % nrows);
      rf[rr][h] = __uint_as_float(dsmem_ld_u32(&cm[h], (uint32_t)rr));
    }
    __syncthreads();
    if (threadIdx.x < S && dsmem_ld_u32(&s_abort, threadIdx.x) != 0) s_bad = 1;
    if (threadIdx.x < nrows) {
      const int h = row_of(threadIdx.x);
      float mx = -INFINITY;
      for (int rr = 0; rr < S; ++rr) mx = fmaxf(mx, rf[rr][h]);
      float ls = 0.0f;
      for (int rr = 0; rr < S; ++rr) {
        const float f = merge_scale(rf[rr][h], mx);
        rf[rr][h] = f;
        ls = fmaf(f, __uint_as_float(dsmem_ld_u32(&cl[h], (uint32_t)rr)), ls);
      }
      // 0 for a row with no keys at all
      const float inv = ls > 0.0f ? 1.0f / ls : 0.0f;
      for (int rr = 0; rr < S; ++rr) rf[rr][h] *= inv;
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    const size_t orow = ((size_t)b * p.Hq + (size_t)g * G) * kHeadDim;
    for (int e = threadIdx.x; e < nrows * (kHeadDim / 4); e += kThreads) {
      const int h = row_of(e / (kHeadDim / 4)), d = 4 * (e % (kHeadDim / 4));
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int rr = 0; rr < S; ++rr) {
        const float f = rf[rr][h];
        const uint4 u = dsmem_ld_v4(&cpart[h][d], (uint32_t)rr);
        acc.x = fmaf(f, __uint_as_float(u.x), acc.x);
        acc.y = fmaf(f, __uint_as_float(u.y), acc.y);
        acc.z = fmaf(f, __uint_as_float(u.z), acc.z);
        acc.w = fmaf(f, __uint_as_float(u.w), acc.w);
      }
      if (bad) acc = make_float4(NAN, NAN, NAN, NAN);
      float* dst = h < 4 ? p.out + orow + (size_t)h * kHeadDim : p.wout + orow + (size_t)(h - 4) * kHeadDim;
      *reinterpret_cast<float4*>(dst + d) = acc;
    }
    if (threadIdx.x == 0) {
      if (C <= p.kc) {
        uint32_t mn = 0xffffffffu;
        for (int rr = 0; rr < S; ++rr) mn = min(mn, dsmem_ld_u32(&s_min, (uint32_t)rr));
        p.n_sel[unit] = C;
        if (p.s_cut) p.s_cut[unit] = (C > 0) ? key_score(mn) : -INFINITY;
      } else {
        p.n_sel[unit] = p.kc;
        if (p.s_cut) p.s_cut[unit] = key_score(T);
      }
    }
  }
  cluster_sync();  // keep shared memory alive until rank 0 has read it
}

template <int NQ, bool WIN>
tf_status launch_draft(const DraftParams& p, int units, int Cmax, cudaStream_t stream) {
  static DeviceCache configured;
  if (!configured.get([] {
        return cudaFuncSetAttribute(retrieval_draft_kernel<NQ, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)draft_smem(kMaxSliceKeys)) == cudaSuccess &&
               cudaFuncSetAttribute(retrieval_draft_kernel<NQ, WIN>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                    1) == cudaSuccess;
      }))
    return TF_ERR_CUDA;
  // Cluster size: the largest S <= 16 (at most one CTA per 64 chunks) for
  // which every unit's cluster is resident at once, as the occupancy query for
  // that cluster shape and slice size reports; at least enough CTAs that every
  // slice fits on chip.  On a GB300 (two CTAs per SM) 36 clusters of 8, 30 of
  // 9 and 14 of 16 are resident at once, so 32 units take S = 8 (256 CTAs on
  // 128 SMs).
  const int need = (Cmax + kMaxSliceKeys - 1) / kMaxSliceKeys;
  if (need > kMaxCluster) return TF_ERR_UNSUPPORTED;
  int most = (Cmax + 63) / 64;
  if (most > kMaxCluster) most = kMaxCluster;
  int S = 0;
  for (int cand_s = most; cand_s >= need && cand_s >= 1; --cand_s) {
    const int sl = (Cmax + cand_s - 1) / cand_s;
    cudaLaunchConfig_t qc = {};
    qc.gridDim = dim3(cand_s, units);
    qc.blockDim = dim3(kThreads);
    qc.dynamicSmemBytes = draft_smem(sl);
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = cand_s;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    qc.attrs = qa;
    qc.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, retrieval_draft_kernel<NQ, WIN>, &qc) != cudaSuccess) {
      (void)cudaGetLastError();  // this shape is not available: try a smaller one
      continue;
    }
    if (clusters >= units) {
      S = cand_s;
      break;
    }
  }
  if (S == 0) S = need < 1 ? 1 : need;  // more units than one wave holds: smallest clusters
  const int slice = (Cmax + S - 1) / S;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = draft_smem(slice);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, retrieval_draft_kernel<NQ, WIN>, p) != cudaSuccess) return TF_ERR_CUDA;
  return launch_status();
}

}  // namespace

TF_DBG_READER(dbg_read_draft)

}  // namespace tf

namespace tf {
namespace {

tf_status draft_entry(const uint16_t* q, const uint16_t* M, const uint16_t* K, const uint16_t* V,
                      const int32_t* seq_lens, int B, int Hq, int Hkv, int Lmax, int D, int chunk, int kc, float scale,
                      int32_t* idx, int32_t* n_sel, float* s_cut, float* out, const float* hint,
                      cudaStream_t stream, float* wout = nullptr, int n_sink = 0, int window = 0) {
  if (!q || !M || !K || !V || !seq_lens || !idx || !n_sel || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || kc <= 0 || Hq % Hkv != 0) return TF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(M) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  if (kc > kMaxList || Hq / Hkv > 4) return TF_ERR_UNSUPPORTED;
  if (B == 0) return TF_OK;
  const int units = B * Hkv;
  if (units > 65535) return TF_ERR_UNSUPPORTED;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;
  DraftParams p{q, M, K, V, seq_lens, Hq, Hkv, Lmax, kc, scale * kLog2e, idx, n_sel, s_cut, out, hint,
                B, (B > 1 && B <= 64) ? 1 : 0};
  p.wout = wout;
  p.n_sink = n_sink;
  p.window = window;
  const int G = Hq / Hkv;
  if (G >= 2 && Lmax > 0) {
    const long long rows_total = (long long)units * Lmax;
    if (rows_total >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
    if (!make_piece_map(&p.mapK, K, rows_total) || !make_piece_map(&p.mapV, V, rows_total)) return TF_ERR_CUDA;
  }
  const int cm = Cmax < 1 ? 1 : Cmax;
  if (wout) {  // two to four heads (the window entry point refuses the rest)
    if (G < 2) return TF_ERR_UNSUPPORTED;
    return G == 2 ? launch_draft<2, true>(p, units, cm, stream) : launch_draft<4, true>(p, units, cm, stream);
  }
  switch (G) {
    case 1: return launch_draft<1, false>(p, units, cm, stream);
    case 2: return launch_draft<2, false>(p, units, cm, stream);
    default: return launch_draft<4, false>(p, units, cm, stream);
  }
}

}  // namespace
}  // namespace tf

extern "C" tf_status tf_retrieval_draft_attn(const uint16_t* q, const uint16_t* M, const uint16_t* K,
                                             const uint16_t* V, const int32_t* seq_lens, int B, int Hq, int Hkv,
                                             int Lmax, int D, int chunk, int kc, float scale, int32_t* idx,
                                             int32_t* n_sel, float* s_cut, float* out, tf_stream_t stream) {
  return tf::draft_entry(q, M, K, V, seq_lens, B, Hq, Hkv, Lmax, D, chunk, kc, scale, idx, n_sel, s_cut, out,
                         nullptr, (cudaStream_t)stream);
}

extern "C" tf_status tf_retrieval_window_draft_attn(const uint16_t* q, const uint16_t* M, const uint16_t* K,
                                                    const uint16_t* V, const int32_t* seq_lens, int B, int Hq,
                                                    int Hkv, int Lmax, int D, int chunk, int kc, float scale,
                                                    const float* cut_hint, int n_sink, int window, int32_t* idx,
                                                    int32_t* n_sel, float* s_cut, float* out, float* wout,
                                                    tf_stream_t stream) {
  using namespace tf;
  if (!wout || !aligned16(wout) || n_sink < 0 || window < 0) return TF_ERR_INVALID_ARG;
  if (Hkv <= 0 || Hq % Hkv != 0) return TF_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  // a CTA lists its selected chunks and its share of the window pieces
  const long long pieces = ((long long)n_sink + kChunk - 1) / kChunk + ((long long)window + kChunk - 1) / kChunk + 1;
  if (G < 2 || G > 4 || (long long)kc + pieces > kMaxList) return TF_ERR_UNSUPPORTED;
  return draft_entry(q, M, K, V, seq_lens, B, Hq, Hkv, Lmax, D, chunk, kc, scale, idx, n_sel, s_cut, out, cut_hint,
                     (cudaStream_t)stream, wout, n_sink, window);
}

extern "C" tf_status tf_retrieval_draft_attn_hinted(const uint16_t* q, const uint16_t* M, const uint16_t* K,
                                                    const uint16_t* V, const int32_t* seq_lens, int B, int Hq,
                                                    int Hkv, int Lmax, int D, int chunk, int kc, float scale,
                                                    const float* cut_hint, int32_t* idx, int32_t* n_sel,
                                                    float* s_cut, float* out, tf_stream_t stream) {
  if (!cut_hint) return TF_ERR_INVALID_ARG;
  return tf::draft_entry(q, M, K, V, seq_lens, B, Hq, Hkv, Lmax, D, chunk, kc, scale, idx, n_sel, s_cut, out,
                         cut_hint, (cudaStream_t)stream);
}
