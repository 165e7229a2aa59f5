// a7 (+ a5) -- full-cache verification attention (Force 3) on the 5th-generation
// tensor cores.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": the target model with the complete KV cache checks every drafted
// candidate in one parallel pass.  The candidates form a chain whose keys sit at
// positions L-T .. L-1, so verify query j sees positions [0, L-T+j].
//
// The whole cache is read once per step, so the kernel is HBM-bound (6 flop/B for
// MHA, 24 flop/B for a GQA group of 4); the tensor cores only have to keep up.
// Per CTA: one (sequence, KV head) unit, one group of <= 32 query rows (the
// GQA heads x gamma+1 tokens; the softmax works on them rounded up to 8) and
// one contiguous key range (split-K).  Warp roles:
//   warp 0    TMA producer: 128-key tiles of K and V (2 x 32 KB, 128-byte
//             swizzle) into a 3-stage shared-memory ring;
//   warp 1    tcgen05 issuer: S^T[key, n] = K Q^T into TMEM (M = 128 keys,
//             N = 16 or 32), then O^T = V^T [P_hi; P_lo]^T into TMEM (M = 128
//             head dims, V read MN-major straight from the TMA tile; the hi
//             and lo bf16 parts of P as separate rows, so one MMA per 16 keys
//             reads V once and leaves P_hi V and P_lo V side by side);
//   warps 2.. softmax, one warpgroup per 8 query rows (1 to 4), on TMEM
//             lane = key (online, log2 domain, rescaled only when the running
//             max grows by > 2^8), P written over the K half of the tile's own
//             stage (K is dead once S exists; the stage goes back to the copy
//             engine after P V), handed over before the O of the previous tile
//             is read back (TMEM lane = head dim) and accumulated in fp32
//             registers.  A stage is held from its copy until P V has read it,
//             so the softmax latency sets how many tiles are in flight: with
//             one warpgroup per 8 rows a GQA group's 24 rows take about as
//             long per tile as MHA's 6.
// S and O are double-buffered in TMEM and P has one buffer per stage, so the
// MMAs of tile t+1 overlap the softmax of tile t.  Splits are merged with the
// log-sum-exp identity by the last CTA of each unit (atomic ticket; the
// splits' partial rows are bulk-copied into its idle ring), or inside a
// thread-block cluster through DSMEM when a unit has at most 4 splits.  Every
// mbarrier wait is bounded; on a timeout the CTA records a nonzero status word
// at the start of the workspace and leaves.
//
// The same kernel (GATHER) serves the retrieval drafter's check of the tiny
// drafter's candidates ("The Three Forces of TriForce": the target model over
// the retrieved KV blocks verifies the drafts): query j sees the valid rows of
// the selected 8-token chunks before the candidates (positions < L-T) and
// candidates 0..j.  A key tile is then sixteen 8-row pieces (the selected
// chunks in list order, then the candidate rows), each one 2 KB box of a 3-D
// tensor map per tensor that lands as the piece's two 1 KB swizzle atoms; the
// softmax warps take every key's position from a per-CTA piece table for the
// masks.  With TREE the candidates form a tree (a parent array) and query j
// sees candidate j and its ancestors; in segment mode the K/V buffers hold a
// window of positions of a longer cache (the offloaded verify streams the cache
// through such windows) and each row's (m, l, O) state is written for a final
// merge.
#include <cuda_bf16.h>

#include "sm100_ptx.cuh"
#include "tf_common.cuh"
#include "tma_host.cuh"

namespace tf {
namespace {

using namespace sm100;

constexpr int kTile = 128;          // keys per tile (MMA M)
constexpr int kStages = 3;          // K/V ring depth
constexpr int kStageBytes = 2 * kTile * kHeadDim * 2;  // K + V tile
constexpr int kSoftmaxThreads = 128;  // one softmax warpgroup: the four TMEM lane quarters
constexpr int kGroupRows = 8;         // query rows per softmax warpgroup
constexpr int kMaxRows = 32;        // query rows per CTA (N <= 32)
constexpr int kPiece = 8;           // rows per gathered piece (one chunk, one swizzle atom)
constexpr int kPiecesPerTile = kTile / kPiece;
constexpr int kMaxTilesPerCta = 16;  // gathered tiles per split (piece table size)
constexpr int kPieceBytes = kPiece * kHeadDim * 2;  // one piece of K (or V): 2 KB
constexpr int kMaxClusterMerge = 4;  // splits merged inside one cluster (more: ticketed merge)
constexpr int kPartStride = 4 + kHeadDim;  // one row's partial state: m, l, 2 unused, O[128]  // most splits merged inside one (portable) cluster
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kLptMaxSeqs = 64;  // longest-first block order for batches up to this size


struct VerifyParams {
  const uint16_t* Q;
  const int32_t* seq_lens;
  float* out;
  int* status;    // workspace status word
  int* tickets;   // [units * ngroups]
  float* part_ml; // [units * ngroups, splits_cap, kMaxRows, 2]
  float* part_o;  // [units * ngroups, splits_cap, kMaxRows, D]
  int Hq, Hkv, Lmax, T, ngroups, splits, splits_cap;
  float scale_log2;
  // gathered mode only
  const int32_t* idx;    // [B * Hkv, kc] selected chunk ids
  const int32_t* n_sel;  // [B * Hkv]
  int kc, tiles_per;     // tiles per split
  int no_cand;           // 1: no candidate rows, every key comes from the selection (decode)
  int cmerge;            // 1: the splits of a unit form a cluster and merge through DSMEM
  // segment mode (contiguous only): the K/V buffers hold positions [pos0,
  // pos0 + Lmax) of caches Ltot long; with part_out set, every row's state
  // (m, l, unnormalised O; kPartStride floats) is written instead of O
  int pos0, Ltot;
  float* part_out;
  // candidate tree [B, T]: parent[b * T + j] is the candidate that j extends
  // (-1: the prefix); null: a chain (parent j - 1)
  const int32_t* parent;
  // contiguous mode: 1 = block row r serves the sequence with the r-th
  // longest context (nseq <= kLptMaxSeqs), 0 = batch order
  int nseq, longest_first;
  // contiguous chain mode, optional: the decode queries [B, Hq, 128] of the
  // streaming drafter's window attention, computed as G extra rows per KV
  // head after the G * T verify rows (keys [0, min(n_sink, L)) and
  // [max(n_sink, L - window), L)), written to wout [B, Hq, 128]
  const uint16_t* wq;
  float* wout;
  int n_sink, window;
};

// Final log-sum-exp merge of a unit's split partials by the CTA that finished
// last, with its idle K/V ring as the staging area.  The splits' O rows (rows x
// 128 fp32, contiguous per split) come in by bulk copies, as many splits per
// batch as fit beside the weights, all in flight at once; meanwhile the
// threads load every split's (m, l), and the weights e^{m_s - m} and row sums
// L are formed; each thread then accumulates float4 columns of the output
// from shared memory and writes them divided by L.
template <int kThreads>
__device__ void merge_staged(const float* __restrict__ ml, const float* __restrict__ o, int S, int rows,
                             uint8_t* ring, uint64_t* bar, float* __restrict__ out, float* __restrict__ part,
                             int* status, float* __restrict__ wout = nullptr, int nvl = kMaxRows) {
  constexpr int kRing = kStages * kStageBytes;
  constexpr int kAcc = (kMaxRows * kHeadDim / 4 + kThreads - 1) / kThreads;  // float4 outputs per thread
  const int tid = threadIdx.x;
  const int nw = S * rows;
  const int wbytes = (int)(((size_t)(2 * nw + 2 * kMaxRows) * sizeof(float) + 1023) & ~size_t(1023));
  float* m_w = reinterpret_cast<float*>(ring + kRing - wbytes);  // [S][rows]: m, then the weights
  float* l_s = m_w + nw;                                          // [S][rows]
  float* L_s = l_s + nw;                                          // [rows]: row sums
  float* M_s = L_s + kMaxRows;                                    // [rows]: max m
  const uint32_t split_bytes = (uint32_t)rows * kHeadDim * sizeof(float);
  const int per_batch = max(1, (kRing - wbytes) / (int)split_bytes);
  auto issue = [&](int sp0) {
    const int nb = min(per_batch, S - sp0);
    mbar_arrive_expect_tx(bar, (uint32_t)nb * split_bytes);
    for (int j = 0; j < nb; ++j)
      bulk_load(ring + (size_t)j * split_bytes, o + (size_t)(sp0 + j) * kMaxRows * kHeadDim, split_bytes, bar);
  };
  if (tid == 0) {
    fence_proxy_async_global();
    issue(0);
  }
  for (int i = tid; i < nw; i += kThreads) {
    const int sp = i / rows, n = i % rows;
    const float2 v = __ldcg(reinterpret_cast<const float2*>(ml) + (size_t)sp * kMaxRows + n);
    m_w[i] = v.x;
    l_s[i] = v.y;
  }
  __syncthreads();
  for (int n = tid; n < rows; n += kThreads) {
    float mx = -INFINITY;
    for (int sp = 0; sp < S; ++sp) mx = fmaxf(mx, m_w[sp * rows + n]);
    float Lsum = 0.0f;
    for (int sp = 0; sp < S; ++sp) {
      const float w = merge_scale(m_w[sp * rows + n], mx);
      m_w[sp * rows + n] = w;
      Lsum = fmaf(w, l_s[sp * rows + n], Lsum);
    }
    L_s[n] = Lsum;
    M_s[n] = mx;
  }
  __syncthreads();
  float4 acc[kAcc];
#pragma unroll
  for (int k = 0; k < kAcc; ++k) acc[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  const int n4 = rows * (kHeadDim / 4);
  bool ok = true;
  for (int sp0 = 0, batch = 0; sp0 < S; sp0 += per_batch, ++batch) {
    const int nb = min(per_batch, S - sp0);
    if (!mbar_wait(bar, batch & 1)) {
      ok = false;  // a bounded wait ran out: report, keep no result
      if (tid == 0) atomicExch(status, 1);
      break;
    }
    const float4* st = reinterpret_cast<const float4*>(ring);
#pragma unroll
    for (int k = 0; k < kAcc; ++k) {
      const int e4 = tid + k * kThreads;
      if (e4 < n4) {
        const int n = e4 / (kHeadDim / 4);
        for (int j = 0; j < nb; ++j) {
          const float w = m_w[(sp0 + j) * rows + n];
          const float4 v = st[(size_t)j * n4 + e4];
          acc[k].x = fmaf(w, v.x, acc[k].x);
          acc[k].y = fmaf(w, v.y, acc[k].y);
          acc[k].z = fmaf(w, v.z, acc[k].z);
          acc[k].w = fmaf(w, v.w, acc[k].w);
        }
      }
    }
    if (sp0 + nb < S) {
      fence_proxy_async_smem();  // these reads of the staging area before the next copies into it
      __syncthreads();
      if (tid == 0) issue(sp0 + nb);
    }
  }
  if (!ok) return;
  if (part) {
    // the unit's state over this segment: max m, row sum L, O relative to m
    for (int n = tid; n < rows; n += kThreads) {
      part[(size_t)n * kPartStride + 0] = M_s[n];
      part[(size_t)n * kPartStride + 1] = L_s[n];
    }
#pragma unroll
    for (int k = 0; k < kAcc; ++k) {
      const int e4 = tid + k * kThreads;
      if (e4 < n4) {
        const int n = e4 / (kHeadDim / 4), d4 = e4 % (kHeadDim / 4);
        reinterpret_cast<float4*>(part + (size_t)n * kPartStride + 4)[d4] = acc[k];
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < kAcc; ++k) {
    const int e4 = tid + k * kThreads;
    if (e4 < n4) {
      const int n = e4 / (kHeadDim / 4), d4 = e4 % (kHeadDim / 4);
      const float Lr = L_s[n];
      const float inv = Lr > 0.0f ? 1.0f / Lr : 0.0f;
      // rows [0, nvl) are contiguous verify rows at out, the rest window rows at wout
      float* dst = n < nvl ? out + (size_t)n * kHeadDim : wout + (size_t)(n - nvl) * kHeadDim;
      reinterpret_cast<float4*>(dst)[d4] = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
    }
  }
}

// NR = query rows the softmax warps work on (the group's rows rounded up to 8):
// 8, 16, 24 or 32.  The MMA shapes follow from it.
template <int NR>
struct Smem {
  static constexpr int kGroups = NR / kGroupRows;                    // softmax warpgroups
  static constexpr int kThreads = 64 + kSoftmaxThreads * kGroups;    // + producer and MMA warps
  static constexpr int kNS = NR <= 16 ? 16 : 32;       // N of S = Q K^T (Q rows, zero-padded)
  static constexpr int kQBytes = 2 * kNS * 128;       // two 64-column halves of [kNS x 128] bf16
  // P of tile t is written over the K half of the tile's own stage: K is dead
  // once S has been computed, and the stage is handed back to the copy engine
  // only after P V has read P.  P holds hi and lo bf16 parts of every row, as
  // the B operand of one MMA per 16 keys (N = kNPV): K-major rows [hi 0..NR-1,
  // lo NR..2NR-1] in two 64-key halves for NR <= 16, else MN-major with one
  // 128-byte swizzled row per key (hi parts in elements 0..31, lo parts in
  // 32..63; 8-key groups 1 KB apart), written as 16-byte vectors.
  static constexpr bool kPMnMajor = NR > 16;
  static constexpr int kNPV = kPMnMajor ? 64 : 2 * NR;
  static constexpr int kLoCol = kPMnMajor ? 32 : NR;   // first lo column of O (and of P)
  static constexpr int kPKeyHalf = kNPV * 128;
  static_assert(2 * kPKeyHalf <= kTile * kHeadDim * 2, "P fits over the K tile");
  // TMEM columns: S of two tiles (32 each), then O of two tiles (kNPV each).
  static constexpr uint32_t kTmemCols = 64 + 2 * kNPV <= 128 ? 128u : 256u;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kBytes = kOffQ + kQBytes;
  static constexpr int kDynamic = kBytes + 1024;     // slack for 1024-byte alignment
  // Cluster merge: a split's (m, l) per row and its O rows [NR x 128] fp32
  // in stage 0, idle once the last O has been read back (every tile landed and
  // was consumed).
  static constexpr int kOffCm = 0;
  static constexpr int kOffCo = 256;
  static_assert(kOffCo + NR * kHeadDim * 4 <= kStageBytes, "cluster merge scratch");
};

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
  uint32_t u;
  memcpy(&u, &v, sizeof(u));
  return u;
}

// Barriers of one softmax warpgroup (id 1 + its index; 0 is the block barrier).
__device__ __forceinline__ bool named_bar_or(uint32_t id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %3, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(kSoftmaxThreads), "r"(id));
  return r != 0;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kSoftmaxThreads) : "memory");
}

// WIN: the G window rows of p.wq follow the G * T verify rows (contiguous
// chain mode only).
template <int NR, bool GATHER, bool TREE = false, bool WIN = false>
__global__ void __launch_bounds__(Smem<NR>::kThreads, 1) verify_umma_kernel(const __grid_constant__ CUtensorMap mapK,
                                                                  const __grid_constant__ CUtensorMap mapV,
                                                                  VerifyParams p) {
  using S = Smem<NR>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages];
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_p_full[2], bar_o_full[2], bar_o_free[2];
  __shared__ __align__(8) uint64_t bar_merge;
  __shared__ uint32_t tmem_base_s;
  __shared__ float red[4][NR];
  __shared__ float alpha_s[2][NR];
  __shared__ int rescaled_s[S::kGroups][2];
  __shared__ int s_last, s_abort;
  __shared__ int s_pstart[GATHER ? kPiecesPerTile * kMaxTilesPerCta : 1];  // first position, -1: none
  __shared__ int s_pcand[GATHER ? kPiecesPerTile * kMaxTilesPerCta : 1];   // 1: candidate rows
  __shared__ uint32_t s_vis[16];  // candidate i -> bit n set: query row n of this CTA sees it

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + S::kOffQ;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ug = blockIdx.y;  // ticket and partial slots: every split of a unit shares them
  const int grp = ug % p.ngroups, g = (ug / p.ngroups) % p.Hkv;
  const int seq_slot = ug / (p.ngroups * p.Hkv);
  const int G = p.Hq / p.Hkv;
  const int nv = G * p.T;                          // verify rows per KV head
  const int rows_all = nv + (WIN ? G : 0);         // + the window rows
  const int row0 = grp * kMaxRows;
  const int rows = min(kMaxRows, rows_all - row0);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_full[i], kSoftmaxThreads * S::kGroups);
      mbar_init(&bar_o_full[i], 1);
      mbar_init(&bar_o_free[i], kSoftmaxThreads * S::kGroups);
    }
    mbar_init(&bar_merge, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, S::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&mapK);
    prefetch_tensormap(&mapV);
  }
  pdl_wait();  // everything above is on-chip set-up that may overlap the previous kernel
  // Ragged batches: CTAs start in about block order, so block row r takes the
  // sequence with the r-th longest context (ties in batch order) and the
  // longest units begin in the first wave instead of stretching the last.
  // Every warp ranks the (at most 64) lengths itself: lane i holds sequences
  // i and i + 32, the lengths go round by shuffles, and the one sequence whose
  // rank is this block row's slot comes out of a ballot (no block barrier).
  int b = seq_slot;
  if (p.longest_first) {
    const int l0 = lane < p.nseq ? clamp_len(p.seq_lens[lane], p.Ltot) : -1;
    const int l1 = lane + 32 < p.nseq ? clamp_len(p.seq_lens[lane + 32], p.Ltot) : -1;
    int r0 = 0, r1 = 0;
    for (int j = 0; j < p.nseq; ++j) {
      const int lj = __shfl_sync(0xffffffffu, j < 32 ? l0 : l1, j & 31);
      r0 += (lj > l0 || (lj == l0 && j < lane)) ? 1 : 0;
      r1 += (lj > l1 || (lj == l1 && j < lane + 32)) ? 1 : 0;
    }
    const unsigned m0 = __ballot_sync(0xffffffffu, lane < p.nseq && r0 == seq_slot);
    const unsigned m1 = __ballot_sync(0xffffffffu, lane + 32 < p.nseq && r1 == seq_slot);
    b = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
  }
  const int unit = b * p.Hkv + g;
  const int L = clamp_len(p.seq_lens[b], p.Ltot);
  // outputs: rows [0, nvl) of this group are verify rows (contiguous from
  // out_row0 in out), the rest window rows (contiguous from wrow0 in wout)
  const int nvl = WIN ? min(max(nv - row0, 0), rows) : rows;
  const size_t out_row0 = ((size_t)b * p.Hq + (size_t)g * G) * p.T + row0;
  const size_t wrow0 = (size_t)b * p.Hq + (size_t)g * G + (size_t)max(row0 + nvl - nv, 0);
  auto out_row = [&](int n) -> float* {
    return (!WIN || n < nvl) ? p.out + (out_row0 + n) * kHeadDim : p.wout + (wrow0 + (n - nvl)) * kHeadDim;
  };

  // key range of this split: whole tiles (contiguous), or tiles of the piece
  // list (gathered: selected chunks, then the candidate rows)
  int k0 = 0, k1 = 0, ntiles = 0;
  const int cstart = p.no_cand ? L : max(0, L - p.T);  // first candidate position
  if (!GATHER) {
    // rows of the buffer (positions pos0 + row) that the sequence holds
    const int nloc = min(max(L - p.pos0, 0), p.Lmax);
    const int tiles_all = (nloc + kTile - 1) / kTile;
    const int tiles_per = (tiles_all + p.splits - 1) / p.splits;
    k0 = blockIdx.x * tiles_per * kTile;
    k1 = min(nloc, k0 + tiles_per * kTile);
    ntiles = k1 > k0 ? (k1 - k0 + kTile - 1) / kTile : 0;
  } else {
    const int C = (L + kChunk - 1) / kChunk;
    const int nsel = min(max(p.n_sel[unit], 0), p.kc);
    const int npieces = nsel + (L - cstart + kPiece - 1) / kPiece;
    const int tiles_all = (npieces + kPiecesPerTile - 1) / kPiecesPerTile;
    const int t0 = blockIdx.x * p.tiles_per;
    ntiles = max(0, min(tiles_all, t0 + p.tiles_per) - t0);
    const int32_t* sel = p.idx + (size_t)unit * p.kc;
    for (int e = tid; e < kPiecesPerTile * ntiles; e += S::kThreads) {
      const int gp = t0 * kPiecesPerTile + e;
      int st = -1, cand = 0;
      if (gp < nsel) {
        const int c = sel[gp];
        if (c >= 0 && c < C) st = c * kChunk;
      } else if (gp < npieces) {
        st = cstart + (gp - nsel) * kPiece;
        cand = 1;
      }
      s_pstart[e] = st;
      s_pcand[e] = cand;
    }
  }
  // Tree: which candidates each query row sees, its own and its ancestors'.
  // Parents outside [0, j) end the walk.
  if (TREE && tid < p.T) {
    uint32_t vis = 0;
    for (int n = 0; n < rows; ++n) {
      int x = (row0 + n) % p.T;
      for (int k = 0; k <= p.T && x >= 0; ++k) {
        if (x == tid) {
          vis |= 1u << n;
          break;
        }
        const int px = p.parent ? p.parent[(size_t)b * p.T + x] : x - 1;
        x = (px >= 0 && px < x) ? px : -1;
      }
    }
    s_vis[tid] = vis;
  }
  // Q rows of this group -> shared memory, [kNS x 128] bf16 in two swizzled halves.
  {
    for (int e = tid; e < S::kNS * 16; e += S::kThreads) {
      const int r = e >> 4, c8 = (e & 15) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < rows) {
        const uint16_t* src =
            (!WIN || r < nvl) ? p.Q + (out_row0 + r) * kHeadDim : p.wq + (wrow0 + (r - nvl)) * kHeadDim;
        v = *reinterpret_cast<const uint4*>(src + c8);
      }
      const uint32_t off = (c8 >> 6) * (S::kNS * 128) + sw128_offset(r, c8 & 63);
      *reinterpret_cast<uint4*>(sQ + off) = v;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;  // columns: S0 [0,32) S1 [32,64) O0 [64,64+2N) O1 [64+2N,64+4N)

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (!GATHER) {
      // lane 0 issues; the other lanes wait at the __syncwarp below so that the
      // warp reaches the block barrier only once lane 0 has left its loop
      if (lane == 0) {
        const int row_base = unit * p.Lmax + k0;
        for (int t = 0; t < ntiles; ++t) {
          const int s = t % kStages;
          if (t >= kStages && !mbar_wait(&bar_empty[s], ((t / kStages) - 1) & 1)) {
            atomicExch(&s_abort, 1);
            break;
          }
          if (*(volatile int*)&s_abort) break;
          uint8_t* sk = smem + s * kStageBytes;
          uint8_t* sv = sk + kTile * kHeadDim * 2;
          const bool in_unit = TF_DBG_OK(k0 + t * kTile >= 0 && k0 + t * kTile < p.Lmax, kDbgTile);
          mbar_arrive_expect_tx(&bar_full[s], in_unit ? kStageBytes : 0u);
          const int y = row_base + t * kTile;
          if (in_unit) {
            tma_load_2d(sk, &mapK, &bar_full[s], 0, y);
            tma_load_2d(sk + 16384, &mapK, &bar_full[s], 64, y);
            tma_load_2d(sv, &mapV, &bar_full[s], 0, y);
            tma_load_2d(sv + 16384, &mapV, &bar_full[s], 64, y);
          }
          // The next tile into L2 now: its copy into the ring waits for a stage
          // to come free, and starting the DRAM read here takes that wait off
          // the ring's turnaround.  (One tile ahead measured best; two to four
          // ahead were slower.)
          if (t >= kStages - 1 && t + 1 < ntiles) {
            const int yn = y + kTile;
            tma_prefetch_2d(&mapK, 0, yn);
            tma_prefetch_2d(&mapK, 64, yn);
            tma_prefetch_2d(&mapV, 0, yn);
            tma_prefetch_2d(&mapV, 64, yn);
          }
        }
      }
      __syncwarp();
    } else {
      // Sixteen pieces per tile, one K box and one V box each, issued by the
      // whole warp after lane 0 has waited for the stage and posted the tile's
      // bytes; the warp steps through the loop together.  A gathered tile is
      // laid out piece by piece: [piece][column half][8 rows x 128 B].
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages;
        bool ok = true;
        if (lane == 0) {
          if (t >= kStages && !mbar_wait(&bar_empty[s], ((t / kStages) - 1) & 1)) {
            atomicExch(&s_abort, 1);
            ok = false;
          }
          if (*(volatile int*)&s_abort) ok = false;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        int st = lane < kPiecesPerTile ? s_pstart[t * kPiecesPerTile + lane] : -1;
        if (st >= 0 && !TF_DBG_OK(st < p.Lmax, kDbgTile)) st = -1;
        const unsigned have = __ballot_sync(0xffffffffu, st >= 0);
        if (lane == 0) mbar_arrive_expect_tx(&bar_full[s], (uint32_t)__popc(have) * (kStageBytes / kPiecesPerTile));
        __syncwarp();
        // lanes 0..15 fetch the K of piece `lane`, lanes 16..31 its V; a piece
        // is one 2 KB box that lands as its two 1 KB swizzle atoms
        const int st_kv = __shfl_sync(0xffffffffu, st, lane & 15);
        if (st_kv >= 0) {
          uint8_t* dst = smem + s * kStageBytes + (lane >> 4) * (kTile * kHeadDim * 2) + (lane & 15) * kPieceBytes;
          tma_load_3d(dst, lane < 16 ? &mapK : &mapV, &bar_full[s], 0, unit * p.Lmax + st_kv, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // lane 0 issues; the __syncwarp below keeps the warp together for the
    // block barrier and the warp-wide TMEM release at the end
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(128, S::kNS, false, false);
      const uint32_t idO = idesc_bf16_f32(128, S::kNPV, true, S::kPMnMajor);
      const uint32_t q_addr = smem_u32(sQ);
      for (int t = 0; t <= ntiles; ++t) {
        if (t < ntiles) {
          const int s = t % kStages;
          if (!mbar_wait(&bar_full[s], (t / kStages) & 1)) { atomicExch(&s_abort, 1); break; }
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // K (M = key, K = head dim), K-major: contiguous tiles hold the two
            // 64-column halves 16 KB apart with 8-key groups 1 KB apart;
            // gathered tiles hold them 1 KB apart with 8-key groups 2 KB apart
            const uint64_t a = GATHER ? smem_desc(k_addr + (kk >> 2) * 1024 + (kk & 3) * 32, 16, kPieceBytes)
                                      : smem_desc(k_addr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc(q_addr + (kk >> 2) * (S::kNS * 128) + (kk & 3) * 32, 16, 1024);
            mma_bf16(tmem + (t & 1) * 32, a, bd, idS, kk > 0);
          }
          mma_commit(&bar_s_full[t & 1]);
        }
        if (t >= 1) {
          const int u = t - 1;
          if (!mbar_wait(&bar_p_full[u & 1], (u >> 1) & 1)) { atomicExch(&s_abort, 1); break; }
          if (u >= 2 && !mbar_wait(&bar_o_free[u & 1], ((u - 2) >> 1) & 1)) { atomicExch(&s_abort, 1); break; }
          tc_fence_after();
          const uint32_t v_addr = smem_u32(smem + (u % kStages) * kStageBytes + kTile * kHeadDim * 2);
          const uint32_t p_addr = smem_u32(smem + (u % kStages) * kStageBytes);  // P over K of tile u
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {
            // A = V^T (M = head dim, K = key), MN-major: 64-dim atoms 16 KB apart
            // and 8-key groups 1 KB apart (contiguous), or 1 KB and 2 KB apart
            // (gathered).  B = P (N = the hi parts of the query rows, then their
            // lo parts; K = key), so one pass over V gives P_hi V and P_lo V in
            // two accumulators.
            const uint64_t a = GATHER ? smem_desc(v_addr + k8 * 2 * kPieceBytes, 1024, kPieceBytes)
                                      : smem_desc(v_addr + k8 * 2048, 16384, 1024);
            const uint64_t bd = S::kPMnMajor
                                    ? smem_desc(p_addr + k8 * 2048, 8192, 1024)
                                    : smem_desc(p_addr + (k8 >> 2) * S::kPKeyHalf + (k8 & 3) * 32, 16, 1024);
            mma_bf16(tmem + 64 + (u & 1) * S::kNPV, a, bd, idO, k8 > 0);
          }
          mma_commit(&bar_o_full[u & 1]);
          mma_commit(&bar_empty[u % kStages]);
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax + correction
    // Warpgroup c (warps 2 + 4c .. 5 + 4c) owns the query rows [8c, 8c + 8);
    // its four warps cover the four TMEM lane quarters.  The warpgroups share
    // nothing but the tile hand-overs, so their chains overlap.
    const int wg = S::kGroups == 1 ? 0 : (warp - 2) >> 2;
    const int nb = wg * kGroupRows;        // first row of this warpgroup
    const uint32_t bar_id = 1u + (uint32_t)wg;
    const int q4 = warp & 3;               // TMEM lane quarter of this warp
    const int my = q4 * 32 + lane;         // key index in the tile / head dim of O
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    constexpr int R = kGroupRows;
    float m_run[R], l_part[R], acc[R];
    int lim[TREE ? 1 : R];  // chain: query row nb + j sees positions <= lim[j]
#pragma unroll
    for (int j = 0; j < R; ++j) {
      m_run[j] = -INFINITY;
      l_part[j] = 0.0f;
      acc[j] = 0.0f;
      if (!TREE) lim[j] = (nb + j < rows) ? (L - p.T + ((row0 + nb + j) % p.T)) : -1;
    }
    // window rows of this warpgroup (bit j: row nb + j) and their two key ranges
    uint32_t wrows = 0;
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (WIN && nb + j >= nvl && nb + j < rows) wrows |= 1u << j;
    const int w_sink = min(p.n_sink, L), w_from = max(p.n_sink, L - p.window);
    // A warpgroup without verify rows (window rows, padding) has P = 0 in
    // every tile that holds no window key: it skips their scores and O.
    auto skip_tile = [&](int t) -> bool {
      if (nb >= rows) return true;
      if (!WIN || nb < nvl) return false;
      const int lo = p.pos0 + k0 + t * kTile;  // contiguous mode: window rows exist only there
      return lo >= w_sink && lo + kTile <= w_from;
    };
    const uint32_t all_rows = rows >= 32 ? 0xffffffffu : ((1u << rows) - 1u);
    const int cbase = L - p.T;  // position of candidate 0
    // Every wait is followed by a vote over the warpgroup so that a timeout
    // makes all of its threads leave the loop together (its named barriers
    // stay matched).
    bool zero_v = false;  // this key row of the tile must be zeroed in V
    for (int t = 0; t <= ntiles; ++t) {
      float sc[R];  // scores, then softmax weights of tile t
      if (t < ntiles) {
        const bool timed_out = !mbar_wait(&bar_s_full[t & 1], (t >> 1) & 1);
        if (named_bar_or(bar_id, timed_out)) {
          if (my == 0) atomicExch(&s_abort, 1);
          break;
        }
        tc_fence_after();
        const bool skip = skip_tile(t);  // uniform over the warpgroup
        if (!skip) {
          tmem_ld8(tmem + (t & 1) * 32 + lane_off + nb, sc);
          tmem_ld_wait();
        }
        // this key's position and whether it may be seen at all; a candidate
        // key (position >= L - T) only by the rows whose candidate extends it
        int pos;
        bool key_ok, chain;
        if (!GATHER) {
          const int row = k0 + t * kTile + my;
          key_ok = row < k1;
          pos = p.pos0 + row;  // position in the sequence
          chain = true;
          zero_v = t == ntiles - 1 && !key_ok;  // rows past the range in the last tile
        } else {
          const int li = t * kPiecesPerTile + (my >> 3);
          const int st = s_pstart[li];
          chain = s_pcand[li] != 0;
          pos = st + (my & 7);
          key_ok = st >= 0 && pos < L && (chain ? pos >= cstart : pos < cstart);
          zero_v = !key_ok;  // rows of empty pieces, past L, or counted elsewhere
        }
        if (skip) {
#pragma unroll
          for (int j = 0; j < R; ++j) sc[j] = 0.0f;
          if (my == 0) rescaled_s[wg][t & 1] = 0;
        } else {
          uint32_t vis = 0;
          if (TREE) {
            const int ci = pos - cbase;
            vis = !key_ok ? 0u : (chain && ci >= 0) ? s_vis[ci < 16 ? ci : 15] : all_rows;
            vis >>= nb;
          }
          bool need = false;
#pragma unroll
          for (int j = 0; j < R; ++j) {
            const bool seen = (WIN && ((wrows >> j) & 1u)) ? (pos < w_sink || pos >= w_from)
                                                            : (!chain || pos <= lim[TREE ? 0 : j]);
            const bool valid = TREE ? ((vis >> j) & 1u) != 0u : (key_ok && seen);
            sc[j] = valid ? sc[j] * p.scale_log2 : -INFINITY;
            need |= sc[j] > m_run[j] + kRescaleThreshold;
          }
          need = named_bar_or(bar_id, need);
          if (need) {
            // tile max per row, then a new reference max for every row that grew
#pragma unroll
            for (int j = 0; j < R; ++j) {
              float v = sc[j];
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
              if (lane == 0) red[q4][nb + j] = v;
            }
            named_bar_sync(bar_id);
#pragma unroll
            for (int j = 0; j < R; ++j) {
              const int n = nb + j;
              const float tmax = fmaxf(fmaxf(red[0][n], red[1][n]), fmaxf(red[2][n], red[3][n]));
              const float mn = fmaxf(m_run[j], tmax);
              const float a = merge_scale(m_run[j], mn);
              l_part[j] *= a;
              if (my == 0) alpha_s[t & 1][n] = a;
              m_run[j] = mn;
            }
            named_bar_sync(bar_id);  // red[] is reused by the next rescale
          }
          if (my == 0) rescaled_s[wg][t & 1] = need ? 1 : 0;
#pragma unroll
          for (int j = 0; j < R; ++j) sc[j] = (sc[j] == -INFINITY) ? 0.0f : exp2f(sc[j] - m_run[j]);
        }
      }
      if (t < ntiles) {
        // P for this tile as hi + lo bf16 parts (P V error ~2^-17 instead of
        // 2^-9 relative).
        uint8_t* pbuf = smem + (t % kStages) * kStageBytes;  // over the K tile
        if constexpr (S::kPMnMajor) {
          // key `my` owns one 128-byte row: 16-byte chunk c < 4 holds the hi
          // parts of rows 8c..8c+7, chunk c + 4 their lo parts; this
          // warpgroup writes chunks wg and wg + 4
          uint8_t* prow = pbuf + (my >> 3) * 1024 + (my & 7) * 128;
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a0 = sc[2 * j], a1 = sc[2 * j + 1];
            l_part[2 * j] += a0;
            l_part[2 * j + 1] += a1;
            const __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(a0 - __low2float(h), a1 - __high2float(h));
            hw[j] = bf16x2_bits(h);
            lw[j] = bf16x2_bits(lo);
          }
          *reinterpret_cast<uint4*>(prow + ((wg ^ (my & 7)) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(prow + (((wg + 4) ^ (my & 7)) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        } else {
          // K-major: row n (hi) and row NR + n (lo), column = key
          const uint32_t off_key = (uint32_t)(my >> 6) * S::kPKeyHalf;
#pragma unroll
          for (int j = 0; j < R; ++j) {
            const int n = nb + j;
            const float pv = sc[j];
            const __nv_bfloat16 hi = __float2bfloat16_rn(pv);
            const __nv_bfloat16 lo = __float2bfloat16_rn(pv - __bfloat162float(hi));
            l_part[j] += pv;
            *reinterpret_cast<__nv_bfloat16*>(pbuf + off_key + sw128_offset(n, my & 63)) = hi;
            *reinterpret_cast<__nv_bfloat16*>(pbuf + off_key + sw128_offset(NR + n, my & 63)) = lo;
          }
        }
        if (zero_v && wg == 0) {
          // Rows nobody may see can hold anything (even NaN): zero them in
          // the V tile so 0 * V stays 0 in the MMA.  Waiting on the (already
          // completed) TMA barrier orders these writes after the tile landed.
          const int s = t % kStages;
          mbar_wait(&bar_full[s], (t / kStages) & 1);
          uint8_t* sv = smem + s * kStageBytes + kTile * kHeadDim * 2;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(sv + (GATHER ? (my >> 3) * kPieceBytes + h * 1024 + (my & 7) * 128
                                                     : h * 16384 + my * 128) +
                                        c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_p_full[t & 1]);
      }
      if (t >= 1) {
        // O of the previous tile, folded in after P of this tile has been
        // handed to the MMA warp (the two use different alpha / rescale slots)
        const int u = t - 1;
        const bool timed_out = !mbar_wait(&bar_o_full[u & 1], (u >> 1) & 1);
        if (named_bar_or(bar_id, timed_out)) {  // also orders alpha_s / rescaled_s of tile u
          if (my == 0) atomicExch(&s_abort, 1);
          break;
        }
        tc_fence_after();
        if (!skip_tile(u)) {  // a skipped tile added P V = 0 to these rows
          float ov[R], ol[R];
          const uint32_t o_col = tmem + 64 + (u & 1) * S::kNPV + lane_off + nb;
          tmem_ld8(o_col, ov);
          tmem_ld8(o_col + S::kLoCol, ol);
          tmem_ld_wait();
          const bool resc = rescaled_s[wg][u & 1] != 0;
#pragma unroll
          for (int j = 0; j < R; ++j) acc[j] = (resc ? acc[j] * alpha_s[u & 1][nb + j] : acc[j]) + (ov[j] + ol[j]);
        }
        tc_fence_before();
        mbar_arrive(&bar_o_free[u & 1]);
      }
    }

    // ---- row sums across the 128 key lanes
#pragma unroll
    for (int j = 0; j < R; ++j) {
      float v = l_part[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[q4][nb + j] = v;
    }
    named_bar_sync(bar_id);
    auto row_sum = [&](int n) { return (red[0][n] + red[1][n]) + (red[2][n] + red[3][n]); };
    if (p.splits == 1 && p.part_out) {
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int n = nb + j;
        if (n < rows) {
          float* pr = p.part_out + (out_row0 + n) * kPartStride;
          if (my == 0) {
            pr[0] = m_run[j];
            pr[1] = row_sum(n);
          }
          pr[4 + my] = acc[j];
        }
      }
    } else if (p.splits == 1) {
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int n = nb + j;
        if (n < rows) {
          const float l = row_sum(n);
          out_row(n)[my] = (l > 0.0f) ? acc[j] / l : 0.0f;
        }
      }
    } else if (p.cmerge) {
      // stage 0 is idle: every MMA (and so every copy) has completed once this
      // warpgroup has read back the last O
      float* cm = reinterpret_cast<float*>(smem + S::kOffCm);
      float* co = reinterpret_cast<float*>(smem + S::kOffCo);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int n = nb + j;
        if (n < rows) {
          if (my == 0) {
            cm[n * 2 + 0] = m_run[j];
            cm[n * 2 + 1] = row_sum(n);
          }
          co[n * kHeadDim + my] = acc[j];
        }
      }
    } else {
      float* ml = p.part_ml + ((size_t)ug * p.splits_cap + blockIdx.x) * kMaxRows * 2;
      float* po = p.part_o + ((size_t)ug * p.splits_cap + blockIdx.x) * kMaxRows * kHeadDim;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int n = nb + j;
        if (n < rows) {
          if (my == 0) {
            ml[n * 2 + 0] = m_run[j];
            ml[n * 2 + 1] = row_sum(n);
          }
          po[n * kHeadDim + my] = acc[j];
        }
      }
    }
  }

  // ---- teardown (all warps)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, S::kTmemCols);
  if (s_abort) {
    if (tid == 0) atomicExch(p.status, 1);
    // Let any TMA copy still in flight land before the CTA's shared memory goes away.
    if (tid == 0)
      for (int s = 0; s < kStages; ++s) mbar_wait(&bar_full[s], 0, 1u << 8);
    if (!p.cmerge) return;  // cluster peers still wait for this CTA at the barriers below
  }
  if (p.splits == 1) return;

  if (p.cmerge) {
    // Every split of the unit has left its partial in shared memory; each rank
    // of the cluster merges its share of the unit's outputs from all of them.
    __shared__ float s_w[kMaxClusterMerge * kMaxRows], s_l[kMaxClusterMerge * kMaxRows], s_L[kMaxRows];
    cluster_sync();
    const int S = p.splits;
    const uint32_t rank = cluster_ctarank();
    const float* cm = reinterpret_cast<const float*>(smem + Smem<NR>::kOffCm);
    const float* co = reinterpret_cast<const float*>(smem + Smem<NR>::kOffCo);
    for (int i = tid; i < S * rows; i += Smem<NR>::kThreads) {
      const int sp = i / rows, n = i % rows;
      s_w[i] = __uint_as_float(dsmem_ld_u32(cm + n * 2 + 0, sp));
      s_l[i] = __uint_as_float(dsmem_ld_u32(cm + n * 2 + 1, sp));
    }
    __syncthreads();
    for (int n = tid; n < rows; n += Smem<NR>::kThreads) {
      float mx = -INFINITY;
      for (int sp = 0; sp < S; ++sp) mx = fmaxf(mx, s_w[sp * rows + n]);
      float Lsum = 0.0f;
      for (int sp = 0; sp < S; ++sp) {
        const float w = merge_scale(s_w[sp * rows + n], mx);
        s_w[sp * rows + n] = w;
        Lsum = fmaf(w, s_l[sp * rows + n], Lsum);
      }
      s_L[n] = Lsum;
    }
    __syncthreads();
    for (int e4 = (int)rank * Smem<NR>::kThreads + tid; e4 < rows * (kHeadDim / 4); e4 += S * Smem<NR>::kThreads) {
      const int n = e4 / (kHeadDim / 4), d = (e4 % (kHeadDim / 4)) * 4;
      uint4 v[kMaxClusterMerge];
#pragma unroll
      for (int sp = 0; sp < kMaxClusterMerge; ++sp)
        if (sp < S) v[sp] = dsmem_ld_v4(co + n * kHeadDim + d, sp);
      float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int sp = 0; sp < kMaxClusterMerge; ++sp) {
        if (sp < S) {
          const float w = s_w[sp * rows + n];
          a.x = fmaf(w, __uint_as_float(v[sp].x), a.x);
          a.y = fmaf(w, __uint_as_float(v[sp].y), a.y);
          a.z = fmaf(w, __uint_as_float(v[sp].z), a.z);
          a.w = fmaf(w, __uint_as_float(v[sp].w), a.w);
        }
      }
      const float Lr = s_L[n];
      const float inv = Lr > 0.0f ? 1.0f / Lr : 0.0f;
      a.x *= inv;
      a.y *= inv;
      a.z *= inv;
      a.w *= inv;
      *reinterpret_cast<float4*>(out_row(n) + d) = a;
    }
    cluster_sync();  // peers keep their shared memory until every rank has read it
    return;
  }

  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&p.tickets[ug], 1) == p.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* ml0 = p.part_ml + (size_t)ug * p.splits_cap * kMaxRows * 2;
  const float* o0 = p.part_o + (size_t)ug * p.splits_cap * kMaxRows * kHeadDim;
  merge_staged<Smem<NR>::kThreads>(ml0, o0, p.splits, rows, smem, &bar_merge, p.out + out_row0 * kHeadDim,
               p.part_out ? p.part_out + out_row0 * kPartStride : nullptr, p.status,
               WIN ? p.wout + wrow0 * kHeadDim : nullptr, nvl);
  if (tid == 0) p.tickets[ug] = 0;
}

// ------------------------------------------------------------------ host side

int verify_splits_cap(int Lmax) {
  int tiles = (Lmax + kTile - 1) / kTile;
  int cap = (tiles + 3) / 4;  // at least 4 tiles per split
  if (cap > 256) cap = 256;
  return cap < 1 ? 1 : cap;
}

// Pick the split count so that (units x groups x splits) CTAs, one per SM,
// fill whole waves with at least 4 tiles per CTA.
int verify_splits(int ug, int Lmax, int sms) {
  const int cap = verify_splits_cap(Lmax);
  int best = 1;
  double best_eff = -1.0;
  for (int waves = 1; waves <= 16; ++waves) {
    int s = (waves * sms + ug / 2) / ug;
    if (s < 1) s = 1;
    if (s > cap) s = cap;
    const long long ctas = (long long)ug * s;
    const long long full = (ctas + sms - 1) / sms * sms;
    const double eff = (double)ctas / (double)full;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
    if (eff > 0.97) break;
  }
  return best;
}

size_t verify_ws(int units, int rows_all, int Lmax) {
  const int ngroups = (rows_all + kMaxRows - 1) / kMaxRows;
  const size_t ug = (size_t)units * ngroups;
  const size_t cap = (size_t)verify_splits_cap(Lmax);
  return 256 + align_up(ug * sizeof(int), 256) + align_up(ug * cap * kMaxRows * 2 * sizeof(float), 256) +
         ug * cap * kMaxRows * kHeadDim * sizeof(float);
}

template <int NR, bool GATHER, bool TREE, bool WIN>
tf_status launch(const CUtensorMap& mk, const CUtensorMap& mv, const VerifyParams& p, dim3 grid,
                 cudaStream_t stream) {
  static DeviceCache configured;
  if (!configured.get([] {
        return cudaFuncSetAttribute(verify_umma_kernel<NR, GATHER, TREE, WIN>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<NR>::kDynamic) == cudaSuccess;
      }))
    return TF_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Smem<NR>::kThreads);
  cfg.dynamicSmemBytes = Smem<NR>::kDynamic;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.cmerge ? (unsigned)p.splits : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.cmerge ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, verify_umma_kernel<NR, GATHER, TREE, WIN>, mk, mv, p) != cudaSuccess)
    return TF_ERR_CUDA;
  return launch_status();
}

// The softmax works on the group's query rows rounded up to 8.
template <bool GATHER, bool TREE = false, bool WIN = false>
tf_status launch_rows(int rows_max, const CUtensorMap& mk, const CUtensorMap& mv, const VerifyParams& p, dim3 grid,
                      cudaStream_t stream) {
  switch ((rows_max + 7) >> 3) {
    case 1: return launch<8, GATHER, TREE, WIN>(mk, mv, p, grid, stream);
    case 2: return launch<16, GATHER, TREE, WIN>(mk, mv, p, grid, stream);
    case 3: return launch<24, GATHER, TREE, WIN>(mk, mv, p, grid, stream);
    default: return launch<32, GATHER, TREE, WIN>(mk, mv, p, grid, stream);
  }
}

// Gathered mode: tiles of the longest possible piece list (kc chunks and at most
// two 8-row pieces of candidates), and the split count from a cost model that
// fits every split count measured on this GPU (kc = 512; 32 and 64 units of 24
// query rows): CTAs run in waves of one per SM, and a CTA costs its tiles plus
// about five tile-times of set-up, first copies, partial write and merge.  The
// cheapest count wins (ties: fewer splits); filling the last wave at any price
// was up to 1.8x slower on 64 units (seven splits of five tiles each).
int sparse_verify_tiles(int kc) { return (kc + 2 + kPiecesPerTile - 1) / kPiecesPerTile; }

constexpr int kSplitCostTiles = 5;

int sparse_verify_splits(int ug, int tiles, int sms) {
  const int lo = (tiles + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
  int best = lo;
  long long best_cost = -1;
  for (int s = lo; s <= tiles; ++s) {
    const long long waves = ((long long)ug * s + sms - 1) / sms;
    const long long cost = waves * (kSplitCostTiles + (tiles + s - 1) / s);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

size_t sparse_verify_ws(int units, int rows_all, int kc) {
  const int ngroups = (rows_all + kMaxRows - 1) / kMaxRows;
  const size_t ug = (size_t)units * ngroups;
  const size_t cap = (size_t)sparse_verify_tiles(kc);
  return 256 + align_up(ug * sizeof(int), 256) + align_up(ug * cap * kMaxRows * 2 * sizeof(float), 256) +
         ug * cap * kMaxRows * kHeadDim * sizeof(float);
}

}  // namespace
TF_DBG_READER(dbg_read_verify)

}  // namespace tf

extern "C" size_t tf_verify_attn_workspace(int B, int Hq, int Hkv, int Lmax, int T) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lmax <= 0 || T <= 0 || Hq % Hkv) return 0;
  return tf::verify_ws(B * Hkv, (Hq / Hkv) * T, Lmax);
}

namespace tf {
namespace {

// The contiguous verify over K/V buffers holding positions [pos0, pos0 + Lmax)
// of caches Ltot long (the whole cache: pos0 = 0, Ltot = Lmax), writing O, or
// each row's partial state to part_out when it is set.  Arguments validated.
tf_status verify_contig(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* seq_lens, int B,
                        int Hq, int Hkv, int Lmax, int T, float scale, float* out, void* ws, cudaStream_t stream,
                        int pos0, int Ltot, float* part_out, const int32_t* parent = nullptr,
                        const uint16_t* wq = nullptr, float* wout = nullptr, int n_sink = 0, int window = 0) {
  const long long rows_total = (long long)B * Hkv * Lmax;
  CUtensorMap mk, mv;
  if (!make_kv_map(&mk, K, rows_total, kTile) || !make_kv_map(&mv, V, rows_total, kTile)) return TF_ERR_CUDA;
  VerifyParams p{};
  const int rows_all = (Hq / Hkv) * T + (wq ? Hq / Hkv : 0);
  p.Q = Q;
  p.seq_lens = seq_lens;
  p.out = out;
  p.wq = wq;
  p.wout = wout;
  p.n_sink = n_sink;
  p.window = window;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lmax = Lmax;
  p.Ltot = Ltot;
  p.pos0 = pos0;
  p.part_out = part_out;
  p.parent = parent;
  p.T = T;
  p.nseq = B;
  p.longest_first = (B > 1 && B <= kLptMaxSeqs) ? 1 : 0;
  p.ngroups = (rows_all + kMaxRows - 1) / kMaxRows;
  p.splits_cap = verify_splits_cap(Lmax);
  const int ug = B * Hkv * p.ngroups;
  p.splits = verify_splits(ug, Lmax, num_sms());
  p.scale_log2 = scale * kLog2e;
  char* w = static_cast<char*>(ws);
  p.status = reinterpret_cast<int*>(w);
  p.tickets = reinterpret_cast<int*>(w + 256);
  p.part_ml = reinterpret_cast<float*>(w + 256 + align_up((size_t)ug * sizeof(int), 256));
  p.part_o = reinterpret_cast<float*>(w + 256 + align_up((size_t)ug * sizeof(int), 256) +
                                      align_up((size_t)ug * p.splits_cap * kMaxRows * 2 * sizeof(float), 256));
  dim3 grid(p.splits, ug);
  const int rows_max = rows_all < kMaxRows ? rows_all : kMaxRows;
  if (wq) return launch_rows<false, false, true>(rows_max, mk, mv, p, grid, stream);
  return parent ? launch_rows<false, true>(rows_max, mk, mv, p, grid, stream)
                : launch_rows<false, false>(rows_max, mk, mv, p, grid, stream);
}

// Log-sum-exp merge of per-segment row states: part [nseg][rows][kPartStride]
// -> out [rows][128].  One warp per row, 4 head dims per lane.
__global__ void __launch_bounds__(256) merge_segments_kernel(const float* __restrict__ part, int nseg, int rows,
                                                             float* __restrict__ out) {
  pdl_wait();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;
  const size_t seg_stride = (size_t)rows * kPartStride;
  const float* pr = part + (size_t)row * kPartStride;
  float mx = -INFINITY;
  for (int sg = 0; sg < nseg; ++sg) mx = fmaxf(mx, __ldg(pr + sg * seg_stride));
  float L = 0.0f;
  float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int sg = 0; sg < nseg; ++sg) {
    const float* ps = pr + sg * seg_stride;
    const float w = merge_scale(__ldg(ps), mx);
    L = fmaf(w, __ldg(ps + 1), L);
    const float4 v = __ldg(reinterpret_cast<const float4*>(ps + 4) + lane);
    o.x = fmaf(w, v.x, o.x);
    o.y = fmaf(w, v.y, o.y);
    o.z = fmaf(w, v.z, o.z);
    o.w = fmaf(w, v.w, o.w);
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  reinterpret_cast<float4*>(out + (size_t)row * kHeadDim)[lane] = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
}

// Workspace of the offloaded verify: [status + split scratch of one segment
// launch][partial states of every segment][two staging slots of K and V].
struct OffloadLayout {
  size_t verify, parts, slot, total;
  int nseg_max;
};

OffloadLayout offload_layout(int B, int Hq, int Hkv, int Lmax, int T, int seg_rows) {
  OffloadLayout o;
  const int units = B * Hkv;
  o.nseg_max = (Lmax + seg_rows - 1) / seg_rows;
  o.verify = align_up(verify_ws(units, (Hq / Hkv) * T, seg_rows), 1024);
  o.parts = align_up((size_t)o.nseg_max * B * Hq * T * kPartStride * sizeof(float), 1024);
  o.slot = align_up((size_t)units * seg_rows * kHeadDim * 2, 1024);  // one tensor's rows of one segment
  o.total = o.verify + o.parts + 4 * o.slot;
  return o;
}

}  // namespace
}  // namespace tf

extern "C" tf_status tf_verify_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                                    const int32_t* seq_lens, int B, int Hq, int Hkv, int Lmax, int D, int T,
                                    float scale, float* out, void* ws, size_t ws_bytes, tf_stream_t stream) {
  using namespace tf;
  if (!Q || !K || !V || !seq_lens || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || Hq % Hkv || T < 1) return TF_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || T > 16) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  const long long rows_total = (long long)B * Hkv * Lmax;
  if (rows_total >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
  const size_t need = verify_ws(B * Hkv, (Hq / Hkv) * T, Lmax);
  if (!ws || ws_bytes < need || !aligned16(ws)) return TF_ERR_WORKSPACE;
  return verify_contig(Q, K, V, seq_lens, B, Hq, Hkv, Lmax, T, scale, out, ws, stream, 0, Lmax, nullptr);
}

namespace tf {
namespace {

// The window rows ride in the verify launch when they change neither the
// number of 32-row groups nor the kernel's row count (rows of the widest
// group rounded up to 8), i.e. when they fill padding rows.  A group of window
// rows alone would re-read the whole cache for a few hundred keys (128K, G = 8,
// T = 4: 212.6 us per layer in one launch, 201.2 us in two), and the 32-row
// kernel (18 warps, so at most 96 registers a thread) in place of the 24-row
// one cost more inside the decode step than the window launch it saves (128K,
// batch 4, G = 4, T = 6: 12.99 against 12.63 ms per step); both get two
// launches.
bool window_rows_fit(int G, int T) {
  auto groups = [](int rows) { return (rows + kMaxRows - 1) / kMaxRows; };
  auto width = [](int rows) { return (min(rows, kMaxRows) + 7) >> 3; };
  return groups(G * (T + 1)) == groups(G * T) && width(G * (T + 1)) == width(G * T);
}

}  // namespace
}  // namespace tf

extern "C" size_t tf_verify_window_attn_workspace(int B, int Hq, int Hkv, int Lmax, int T, int n_sink, int window) {
  using namespace tf;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lmax <= 0 || T < 1 || n_sink < 0 || window < 0 || Hq % Hkv) return 0;
  const int G = Hq / Hkv;
  if (window_rows_fit(G, T)) return verify_ws(B * Hkv, G * (T + 1), Lmax);
  return align_up(verify_ws(B * Hkv, G * T, Lmax), 256) + tf_stream_window_attn_workspace(B, Hq, Hkv, n_sink, window);
}

extern "C" tf_status tf_verify_window_attn(const uint16_t* Q, const uint16_t* q, const uint16_t* K,
                                           const uint16_t* V, const int32_t* seq_lens, int B, int Hq, int Hkv,
                                           int Lmax, int D, int T, int n_sink, int window, float scale,
                                           float* out, float* wout, void* ws, size_t ws_bytes,
                                           tf_stream_t stream) {
  using namespace tf;
  if (!Q || !q || !K || !V || !seq_lens || !out || !wout) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || Hq % Hkv || T < 1 || n_sink < 0 || window < 0)
    return TF_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) || !aligned16(wout))
    return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || T > 16) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  const long long rows_total = (long long)B * Hkv * Lmax;
  if (rows_total >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (!window_rows_fit(G, T)) {
    const size_t vneed = align_up(verify_ws(B * Hkv, G * T, Lmax), 256);
    if (!ws || ws_bytes < vneed || !aligned16(ws)) return TF_ERR_WORKSPACE;
    const tf_status st = tf_stream_window_attn(q, K, V, seq_lens, B, Hq, Hkv, Lmax, D, n_sink, window, scale, wout,
                                               static_cast<char*>(ws) + vneed, ws_bytes - vneed, stream);
    if (st != TF_OK) return st;
    return verify_contig(Q, K, V, seq_lens, B, Hq, Hkv, Lmax, T, scale, out, ws, stream, 0, Lmax, nullptr);
  }
  const size_t need = verify_ws(B * Hkv, G * (T + 1), Lmax);
  if (!ws || ws_bytes < need || !aligned16(ws)) return TF_ERR_WORKSPACE;
  return verify_contig(Q, K, V, seq_lens, B, Hq, Hkv, Lmax, T, scale, out, ws, stream, 0, Lmax, nullptr, nullptr,
                       q, wout, n_sink, window);
}

extern "C" tf_status tf_verify_attn_tree(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                                         const int32_t* seq_lens, const int32_t* parent, int B, int Hq, int Hkv,
                                         int Lmax, int D, int T, float scale, float* out, void* ws, size_t ws_bytes,
                                         tf_stream_t stream) {
  using namespace tf;
  if (!parent) return TF_ERR_INVALID_ARG;
  if (!Q || !K || !V || !seq_lens || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || Hq % Hkv || T < 1) return TF_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || T > 16) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  if ((long long)B * Hkv * Lmax >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
  const size_t need = verify_ws(B * Hkv, (Hq / Hkv) * T, Lmax);
  if (!ws || ws_bytes < need || !aligned16(ws)) return TF_ERR_WORKSPACE;
  return verify_contig(Q, K, V, seq_lens, B, Hq, Hkv, Lmax, T, scale, out, ws, stream, 0, Lmax, nullptr, parent);
}

extern "C" size_t tf_verify_attn_offload_workspace(int B, int Hq, int Hkv, int Lmax, int T, int seg_rows) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lmax <= 0 || T <= 0 || Hq % Hkv || seg_rows <= 0) return 0;
  return tf::offload_layout(B, Hq, Hkv, Lmax, T, seg_rows).total;
}

extern "C" tf_status tf_verify_attn_offload(const uint16_t* Q, const uint16_t* K_host, const uint16_t* V_host,
                                            const int32_t* seq_lens, int L_stream, int B, int Hq, int Hkv, int Lmax,
                                            int D, int T, float scale, float* out, int seg_rows, void* ws,
                                            size_t ws_bytes, tf_stream_t stream, tf_stream_t copy_stream) {
  using namespace tf;
  if (!Q || !K_host || !V_host || !seq_lens || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || Hq % Hkv || T < 1 || seg_rows <= 0) return TF_ERR_INVALID_ARG;
  if (L_stream < 0 || L_stream > Lmax) return TF_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || T > 16) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  if ((long long)B * Hkv * seg_rows >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
  const OffloadLayout lay = offload_layout(B, Hq, Hkv, Lmax, T, seg_rows);
  if (!ws || ws_bytes < lay.total || !aligned16(ws)) return TF_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream), xs = static_cast<cudaStream_t>(copy_stream);
  char* w = static_cast<char*>(ws);
  float* parts = reinterpret_cast<float*>(w + lay.verify);
  uint16_t* stage[2][2];  // [slot][K, V]
  for (int sl = 0; sl < 2; ++sl)
    for (int kv = 0; kv < 2; ++kv)
      stage[sl][kv] = reinterpret_cast<uint16_t*>(w + lay.verify + lay.parts + (size_t)(2 * sl + kv) * lay.slot);
  const int units = B * Hkv;
  const int rows = B * Hq * T;
  const int nseg = L_stream > 0 ? (L_stream + seg_rows - 1) / seg_rows : 1;
  const size_t row_bytes = (size_t)kHeadDim * 2;

  cudaEvent_t start, copied[2], computed[2];
  if (cudaEventCreateWithFlags(&start, cudaEventDisableTiming) != cudaSuccess) return TF_ERR_CUDA;
  for (int sl = 0; sl < 2; ++sl) {
    cudaEventCreateWithFlags(&copied[sl], cudaEventDisableTiming);
    cudaEventCreateWithFlags(&computed[sl], cudaEventDisableTiming);
  }
  tf_status st = TF_OK;
  // the staging slots may still be read by earlier work on the compute stream
  if (cudaEventRecord(start, cs) != cudaSuccess || cudaStreamWaitEvent(xs, start, 0) != cudaSuccess) st = TF_ERR_CUDA;
  for (int sg = 0; sg < nseg && st == TF_OK; ++sg) {
    const int sl = sg & 1;
    const int pos0 = sg * seg_rows;
    const int n = L_stream > 0 ? (L_stream - pos0 < seg_rows ? L_stream - pos0 : seg_rows) : 0;
    if (sg >= 2 && cudaStreamWaitEvent(xs, computed[sl], 0) != cudaSuccess) st = TF_ERR_CUDA;
    // one copy per tensor: rows [pos0, pos0 + n) of every (b, g) unit
    for (int kv = 0; kv < 2 && st == TF_OK && n > 0; ++kv) {
      const uint16_t* src = (kv == 0 ? K_host : V_host) + (size_t)pos0 * kHeadDim;
      if (cudaMemcpy2DAsync(stage[sl][kv], (size_t)seg_rows * row_bytes, src, (size_t)Lmax * row_bytes,
                            (size_t)n * row_bytes, (size_t)units, cudaMemcpyHostToDevice, xs) != cudaSuccess)
        st = TF_ERR_CUDA;
    }
    if (st == TF_OK && (cudaEventRecord(copied[sl], xs) != cudaSuccess || cudaStreamWaitEvent(cs, copied[sl], 0) != cudaSuccess))
      st = TF_ERR_CUDA;
    if (st == TF_OK)
      st = verify_contig(Q, stage[sl][0], stage[sl][1], seq_lens, B, Hq, Hkv, seg_rows, T, scale, out, ws, cs, pos0,
                         L_stream, parts + (size_t)sg * rows * kPartStride);
    if (st == TF_OK && cudaEventRecord(computed[sl], cs) != cudaSuccess) st = TF_ERR_CUDA;
  }
  if (st == TF_OK) {
    if (launch_pdl(merge_segments_kernel, dim3((rows + 7) / 8), dim3(256), 0, cs, (const float*)parts, nseg, rows,
                   out) != cudaSuccess)
      st = TF_ERR_CUDA;
    else
      st = launch_status();
  }
  cudaEventDestroy(start);
  for (int sl = 0; sl < 2; ++sl) {
    cudaEventDestroy(copied[sl]);
    cudaEventDestroy(computed[sl]);
  }
  return st;
}

extern "C" size_t tf_sparse_verify_attn_workspace(int B, int Hq, int Hkv, int kc, int T) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || kc <= 0 || T <= 0 || Hq % Hkv) return 0;
  return tf::sparse_verify_ws(B * Hkv, (Hq / Hkv) * T, kc);
}

namespace tf {

// The gathered verify over the selected chunks for T query rows per head
// (arguments validated): with candidates (level-1 verification) or, no_cand,
// the decode attention of the retrieval drafter (T = 1, every key from the
// selection).
tf_status sparse_gather(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* seq_lens,
                        const int32_t* idx, const int32_t* n_sel, int B, int Hq, int Hkv, int Lmax, int kc, int T,
                        float scale, float* out, void* ws, cudaStream_t stream, int no_cand) {
  const long long rows_total = (long long)B * Hkv * Lmax;
  CUtensorMap mk, mv;
  if (!make_piece_map(&mk, K, rows_total) || !make_piece_map(&mv, V, rows_total)) return TF_ERR_CUDA;
  VerifyParams p{};
  const int rows_all = (Hq / Hkv) * T;
  p.Q = Q;
  p.seq_lens = seq_lens;
  p.out = out;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lmax = Lmax;
  p.Ltot = Lmax;
  p.T = T;
  p.ngroups = (rows_all + kMaxRows - 1) / kMaxRows;
  p.idx = idx;
  p.n_sel = n_sel;
  p.kc = kc;
  p.no_cand = no_cand;
  const int tiles = sparse_verify_tiles(kc);
  p.splits_cap = tiles;
  const int ug = B * Hkv * p.ngroups;
  p.splits = sparse_verify_splits(ug, tiles, num_sms());
  p.tiles_per = (tiles + p.splits - 1) / p.splits;
  // Splits merge inside a cluster only up to four: clusters of five to seven
  // one-SM CTAs packed badly (up to 1.6x slower than the ticketed merge).
  p.cmerge = (p.splits > 1 && p.splits <= kMaxClusterMerge) ? 1 : 0;
  p.scale_log2 = scale * kLog2e;
  char* w = static_cast<char*>(ws);
  p.status = reinterpret_cast<int*>(w);
  p.tickets = reinterpret_cast<int*>(w + 256);
  p.part_ml = reinterpret_cast<float*>(w + 256 + align_up((size_t)ug * sizeof(int), 256));
  p.part_o = reinterpret_cast<float*>(w + 256 + align_up((size_t)ug * sizeof(int), 256) +
                                      align_up((size_t)ug * p.splits_cap * kMaxRows * 2 * sizeof(float), 256));
  dim3 grid(p.splits, ug);
  const int rows_max = rows_all < kMaxRows ? rows_all : kMaxRows;
  return launch_rows<true>(rows_max, mk, mv, p, grid, stream);
}

size_t sparse_decode_umma_ws(int B, int Hq, int Hkv, int kc) { return sparse_verify_ws(B * Hkv, Hq / Hkv, kc); }

tf_status sparse_decode_umma(const uint16_t* q, const uint16_t* K, const uint16_t* V, const int32_t* seq_lens,
                             const int32_t* idx, const int32_t* n_sel, int B, int Hq, int Hkv, int Lmax, int kc,
                             float scale, float* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if ((long long)B * Hkv * Lmax >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < sparse_decode_umma_ws(B, Hq, Hkv, kc) || !aligned16(ws)) return TF_ERR_WORKSPACE;
  return sparse_gather(q, K, V, seq_lens, idx, n_sel, B, Hq, Hkv, Lmax, kc, 1, scale, out, ws, stream, 1);
}

}  // namespace tf

extern "C" tf_status tf_sparse_verify_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                                           const int32_t* seq_lens, const int32_t* idx, const int32_t* n_sel, int B,
                                           int Hq, int Hkv, int Lmax, int D, int chunk, int kc, int T, float scale,
                                           float* out, void* ws, size_t ws_bytes, tf_stream_t stream) {
  using namespace tf;
  if (!Q || !K || !V || !seq_lens || !idx || !n_sel || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || Hq % Hkv || T < 1 || kc <= 0) return TF_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk || T > 16) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  const long long rows_total = (long long)B * Hkv * Lmax;
  if (rows_total >= (1ll << 31)) return TF_ERR_UNSUPPORTED;
  const size_t need = sparse_verify_ws(B * Hkv, (Hq / Hkv) * T, kc);
  if (!ws || ws_bytes < need || !aligned16(ws)) return TF_ERR_WORKSPACE;

  return sparse_gather(Q, K, V, seq_lens, idx, n_sel, B, Hq, Hkv, Lmax, kc, T, scale, out, ws, stream, 0);
}
