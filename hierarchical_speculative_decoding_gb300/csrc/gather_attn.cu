// a4, a6 (+ a5) -- decode attention over a gathered set of KV positions.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce":
//   Force 2 (retrieval drafter): the target model attends only to the KV
//     blocks retrieved by key-query similarity (the selected chunk list);
//   Force 1 (streaming drafter): attention sinks plus the most recent window.
// Both are one query token per head attending to a small, irregular subset of
// a long cache.  Both are served by one kernel whose unit of work is an 8-row
// "chunk" of K and V: a selected chunk id, or a piece of the sink / window
// ranges (the sinks form one chunk, the window is cut into 8-row pieces).
//
// Design (HBM-bound, ~1 flop/byte; latency matters because a layer moves only
// 64 MiB): split-K over the chunk list.  A producer warp stages chunks into a
// 16-slot shared-memory ring with untiled bulk copies (cp.async.bulk: a chunk's
// K rows and V rows are each one contiguous run of n x 256 bytes; mbarrier
// complete-tx), chunk ids resolved 32 at a time so no copy waits on an id;
// only one lane of the producer warp ever waits on a barrier.
// Four compute warps take chunks in turn: lane (row r, quarter dq) forms
// 32-dim partial dot products, visiting its four 16-byte pieces in a rotated
// order that keeps the shared-memory reads conflict-free; the row score is
// reduced over the 4 quarters, the online softmax runs in the log2 domain in
// fp32, and for P V each lane owns 4 head dims across all rows.  Warps merge in
// shared memory; splits merge with the log-sum-exp identity in the last CTA of
// each unit to finish (atomic ticket, no waiting).  All waits are bounded; a
// timeout (only a hardware fault can cause one) leaves NaN in the outputs.
#include "gather_attn.cuh"
#include "sm100_ptx.cuh"

namespace tf {

using namespace sm100;

constexpr int kComputeWarps = 4;
constexpr int kSlots = 16;
constexpr int kSlotBytes = 4096;  // K rows [0, 2 KB), V rows [2 KB, 4 KB)
constexpr int kGatherSmem = kSlots * kSlotBytes + 128;  // + alignment slack
constexpr int kMaxClusterSplits = 8;  // splits merged inside one (portable) cluster
constexpr int kWindowSplits = 4;      // splits of a window call
// Chunk k sits in slot k % 16 and is consumed by compute warp k % 4: every use
// of a slot is consumed by the same warp, so a phase-parity wait never runs two
// phases ahead of its barrier.
static_assert(kSlots % kComputeWarps == 0, "a slot must always be consumed by the same warp");

// The i-th chunk of a unit's position set: first position y and valid rows n.
template <int MODE>
__device__ __forceinline__ void chunk_at(int e, const int32_t* sel, int C, int L, int has_sink, int ns_eff, int w0,
                                         int& y, int& n) {
  if (MODE == kModeChunks) {
    const int c = sel[e];
    const bool ok = c >= 0 && c < C;
    y = ok ? c * kChunk : 0;
    n = ok ? min(kChunk, L - c * kChunk) : 0;
  } else {
    if (has_sink && e == 0) {
      y = 0;
      n = ns_eff;
    } else {
      y = w0 + (e - has_sink) * kChunk;
      n = min(kChunk, L - y);
    }
  }
}

template <int NQ, int MODE>
__global__ void __launch_bounds__(kGatherThreads, 1) gather_attn_kernel(GatherParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kSlots], bar_empty[kSlots];
  __shared__ int slot_n[kSlots];
  __shared__ float sm_m[kComputeWarps][NQ], sm_l[kComputeWarps][NQ];
  __shared__ float sm_o[kComputeWarps][NQ][kHeadDim];
  __shared__ int s_last, s_abort, s_issued;
  __shared__ float c_m[NQ], c_l[NQ], c_o[NQ][kHeadDim];  // this split's state (cluster merge)
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

  const int unit_grp = blockIdx.y;
  const int unit = unit_grp / p.ngroups, grp = unit_grp % p.ngroups;
  const int b = unit / p.Hkv, g = unit % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = G - grp * NQ < NQ ? G - grp * NQ : NQ;  // heads of this group
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    s_abort = 0;
    s_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  const int L = clamp_len(p.seq_lens[b], p.Lmax);
  const int C = (L + kChunk - 1) / kChunk;

  // ---- this CTA's slice of the unit's chunk list.  For the chunk list the
  // slice bounds come from kc alone, so the ids and n_sel load together.
  int nch = 0, ns_eff = 0, w0 = 0, has_sink = 0, per = 0;
  const int32_t* sel = nullptr;
  if (MODE == kModeChunks) {
    sel = p.idx + (size_t)unit * p.kc;
    per = (p.kc + p.splits - 1) / p.splits;
    nch = p.n_sel[unit];
    nch = nch < 0 ? 0 : (nch > p.kc ? p.kc : nch);
  } else {
    ns_eff = min(p.n_sink, L);
    w0 = max(p.n_sink, L - p.window);
    has_sink = ns_eff > 0 ? 1 : 0;
    nch = has_sink + (max(0, L - w0) + kChunk - 1) / kChunk;
    per = (nch + p.splits - 1) / p.splits;
  }
  const int e0 = blockIdx.x * per;
  const int cnt = max(0, min(nch, e0 + per) - e0);

  if (warp == kComputeWarps) {
    // ---------------------------------------------------------------- producer
    // Chunk positions are resolved 32 at a time, one per lane.  The first use
    // of every ring slot needs no wait, so those lanes issue at once; every
    // later chunk is issued in order by lane 0 alone, so that no two lanes of
    // this warp ever wait on different barriers (diverged lanes need not be
    // scheduled fairly, and a wait that starves another lane could time out).
    const uint16_t* Ku = p.K + (size_t)unit * p.Lmax * kHeadDim;
    const uint16_t* Vu = p.V + (size_t)unit * p.Lmax * kHeadDim;
    auto issue = [&](int slot, int y, int n) {
      if (!TF_DBG_OK(n == 0 || (y >= 0 && n <= kChunk && y + n <= L && L <= p.Lmax), kDbgCacheRow)) n = 0;
      slot_n[slot] = n;
      uint8_t* dst = ring + slot * kSlotBytes;
      const uint32_t bytes = (uint32_t)n * kHeadDim * 2;
      mbar_arrive_expect_tx(&bar_full[slot], 2 * bytes);
      if (n > 0) {
        bulk_load(dst, Ku + (size_t)y * kHeadDim, bytes, &bar_full[slot]);
        bulk_load(dst + 2048, Vu + (size_t)y * kHeadDim, bytes, &bar_full[slot]);
      }
    };
    int issued = 0;  // chunks [0, issued) have been staged
    for (int base = 0; base < cnt; base += 32) {
      int y = 0, n = 0;
      if (base + lane < cnt) chunk_at<MODE>(e0 + base + lane, sel, C, L, has_sink, ns_eff, w0, y, n);
      if (base + lane < cnt && base + lane < kSlots) issue(base + lane, y, n);
      bool ok = true;
      for (int t = 0; t < 32 && base + t < cnt; ++t) {  // warp-uniform
        const int k = base + t;
        const int yk = __shfl_sync(0xffffffffu, y, t), nk = __shfl_sync(0xffffffffu, n, t);
        if (k >= kSlots) {
          if (lane == 0) {
            ok = mbar_wait(&bar_empty[k % kSlots], (k / kSlots - 1) & 1);
            if (ok) issue(k % kSlots, yk, nk);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        issued = k + 1;
      }
      if (!ok) {
        if (lane == 0) atomicExch(&s_abort, 1);
        break;
      }
    }
    if (lane == 0) s_issued = issued;
  } else {
    // ---------------------------------------------------------------- compute warps
    // Score phase: lane = (row r, quarter dq) reads 16-byte pieces j of dims
    // [32 dq, 32 dq + 32) in the rotated order jr(j) (conflict-free banks).
    const int r = lane >> 2, dq = lane & 3;
    const int rot = (dq >> 1) + 2 * (r & 1);
    float qv[NQ][32];
#pragma unroll
    for (int h = 0; h < NQ; ++h) {
      const bool on = h < rows;
      const uint16_t* qrow = p.q + ((size_t)b * p.Hq + (size_t)g * G + grp * NQ + (on ? h : 0)) * kHeadDim + dq * 32;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jr = (j + rot) & 3;
        float f[8];
        unpack8(on ? *reinterpret_cast<const uint4*>(qrow + jr * 8) : make_uint4(0, 0, 0, 0), f);
#pragma unroll
        for (int d = 0; d < 8; ++d) qv[h][j * 8 + d] = f[d] * p.scale_log2;
      }
    }
    float m[NQ], l[NQ], o[NQ][4];
#pragma unroll
    for (int h = 0; h < NQ; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[h][i] = 0.0f;
    }
    for (int k = warp; k < cnt; k += kComputeWarps) {
      const int slot = k % kSlots;
      if (!mbar_wait(&bar_full[slot], (k / kSlots) & 1)) {
        if (lane == 0) atomicExch(&s_abort, 1);
        break;
      }
      const int n = slot_n[slot];
      const uint8_t* kb = ring + slot * kSlotBytes;
      const uint8_t* vb = kb + 2048;
      float s[NQ], s4[NQ][4];  // four independent partial sums per head (short FMA chains)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jr = (j + rot) & 3;
        const uint4 kv = *reinterpret_cast<const uint4*>(kb + r * 256 + dq * 64 + jr * 16);
        float f[8];
        unpack8(kv, f);
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          float a = qv[h][j * 8] * f[0];
#pragma unroll
          for (int d = 1; d < 8; ++d) a = fmaf(qv[h][j * 8 + d], f[d], a);
          s4[h][j] = a;
        }
      }
#pragma unroll
      for (int h = 0; h < NQ; ++h) s[h] = (s4[h][0] + s4[h][1]) + (s4[h][2] + s4[h][3]);
      const bool valid = r < n;
#pragma unroll
      for (int h = 0; h < NQ; ++h) {
        s[h] += __shfl_xor_sync(0xffffffffu, s[h], 1);
        s[h] += __shfl_xor_sync(0xffffffffu, s[h], 2);
        s[h] = valid ? s[h] : -INFINITY;
      }
      float pr[NQ];
#pragma unroll
      for (int h = 0; h < NQ; ++h) {
        float cm = s[h];
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
        const float mn = fmaxf(m[h], cm);
        const float alpha = merge_scale(m[h], mn);
        pr[h] = (s[h] == -INFINITY) ? 0.0f : exp2f(s[h] - mn);
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
      for (int rr = 0; rr < n; ++rr) {
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_empty[slot]);
    }
#pragma unroll
    for (int h = 0; h < NQ; ++h) {
      if (lane == 0) {
        sm_m[warp][h] = m[h];
        sm_l[warp][h] = l[h];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sm_o[warp][h][lane * 4 + i] = o[h][i];
    }
  }
  __syncthreads();
  if (s_abort && threadIdx.x == 0) {
    // (only after a timeout) let every copy still in flight land before the
    // ring is reused or the CTA exits
    for (int sl = 0; sl < kSlots && sl < s_issued; ++sl) {
      const int klast = sl + (s_issued - 1 - sl) / kSlots * kSlots;
      mbar_wait(&bar_full[sl], (klast / kSlots) & 1, 1u << 8);
    }
  }
  __syncthreads();

  // ---- merge the compute warps: thread handles (h, d) pairs
  const bool bad = s_abort != 0;
  float* part_ml = p.part_ml + ((size_t)unit_grp * p.splits_cap + blockIdx.x) * NQ * 2;
  float* part_o = p.part_o + ((size_t)unit_grp * p.splits_cap + blockIdx.x) * NQ * kHeadDim;
  for (int e = threadIdx.x; e < rows * kHeadDim; e += kGatherThreads) {
    const int h = e / kHeadDim, d = e % kHeadDim;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) mx = fmaxf(mx, sm_m[w][h]);
    float ls = 0.0f, os = 0.0f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) {
      const float f = merge_scale(sm_m[w][h], mx);
      ls = fmaf(f, sm_l[w][h], ls);
      os = fmaf(f, sm_o[w][h][d], os);
    }
    if (bad) os = NAN;
    if (p.splits == 1) {
      p.out[((size_t)b * p.Hq + (size_t)g * G + grp * NQ + h) * kHeadDim + d] =
          (ls > 0.0f) ? os / ls : (bad ? NAN : 0.0f);
    } else if (p.cmerge) {
      if (d == 0) {
        c_m[h] = mx;
        c_l[h] = ls;
      }
      c_o[h][d] = os;
    } else {
      if (d == 0) {
        part_ml[h * 2 + 0] = mx;
        part_ml[h * 2 + 1] = ls;
      }
      part_o[h * kHeadDim + d] = os;
    }
  }
  if (p.splits == 1) return;

  if (p.cmerge) {
    // The splits of this (unit, group) are one cluster: after a cluster
    // barrier each rank merges its share of the outputs from every rank's
    // state through DSMEM (log-sum-exp identity); a second barrier keeps the
    // states alive until every rank has read them.
    cluster_sync();
    const int S = p.splits;
    const uint32_t rank = cluster_ctarank();
    bool bad_any = false;
    for (int rr = 0; rr < S; ++rr) bad_any |= dsmem_ld_u32(&s_abort, (uint32_t)rr) != 0;
    float* outp = p.out + ((size_t)b * p.Hq + (size_t)g * G + grp * NQ) * kHeadDim;
    for (int e = (int)rank * kGatherThreads + threadIdx.x; e < rows * kHeadDim; e += S * kGatherThreads) {
      const int h = e / kHeadDim, d = e % kHeadDim;
      float mr[8];
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) mr[rr] = rr < S ? __uint_as_float(dsmem_ld_u32(&c_m[h], (uint32_t)rr)) : -INFINITY;
      float mx = -INFINITY;
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) mx = fmaxf(mx, mr[rr]);
      float ls = 0.0f, os = 0.0f;
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        if (rr < S) {
          const float f = merge_scale(mr[rr], mx);
          ls = fmaf(f, __uint_as_float(dsmem_ld_u32(&c_l[h], (uint32_t)rr)), ls);
          os = fmaf(f, __uint_as_float(dsmem_ld_u32(&c_o[h][d], (uint32_t)rr)), os);
        }
      }
      outp[h * kHeadDim + d] = bad_any ? NAN : (ls > 0.0f ? os / ls : 0.0f);
    }
    cluster_sync();
    return;
  }

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&p.tickets[unit_grp], 1) == p.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const float* ml0 = p.part_ml + (size_t)unit_grp * p.splits_cap * NQ * 2;
  const float* o0 = p.part_o + (size_t)unit_grp * p.splits_cap * NQ * kHeadDim;
  float* outp = p.out + ((size_t)b * p.Hq + (size_t)g * G + grp * NQ) * kHeadDim;
  // The chunk ring is idle now: it serves as the merge scratch.
  merge_splits(ml0, o0, p.splits, rows, NQ, reinterpret_cast<float*>(ring),
               [&](int h, int d, float v) { outp[h * kHeadDim + d] = v; });
  if (threadIdx.x == 0) p.tickets[unit_grp] = 0;
}

// ------------------------------------------------------------------ host side

int gather_nq(int rows) {
  if (rows <= 1) return 1;
  if (rows <= 2) return 2;
  return 4;
}

// Chunk-list length bound: P_max positions in 8-row chunks plus the sink chunk.
static int gather_max_chunks(int P_max) { return (P_max + kChunk - 1) / kChunk + 1; }

int gather_splits_cap(int P_max) {
  int s = (gather_max_chunks(P_max) + 3) / 4;  // at least 4 chunks per split
  if (s > 256) s = 256;
  return s < 1 ? 1 : s;
}

size_t gather_workspace(int units, int rows, int P_max) {
  const int nq = gather_nq(rows);
  const int ngroups = (rows + nq - 1) / nq;
  const size_t ug = (size_t)units * ngroups;
  const size_t cap = (size_t)gather_splits_cap(P_max);
  return align_up(ug * sizeof(int), 256) + align_up(ug * cap * nq * 2 * sizeof(float), 256) +
         ug * cap * nq * kHeadDim * sizeof(float);
}

template <int NQ, int MODE>
static int configure() {
  static DeviceCache per_sm;  // resident CTAs per SM on each device, 0 if the setup failed
  return per_sm.get([] {
    if (cudaFuncSetAttribute(gather_attn_kernel<NQ, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGatherSmem) != cudaSuccess)
      return 0;
    return occupancy_blocks((const void*)gather_attn_kernel<NQ, MODE>, kGatherThreads, kGatherSmem);
  });
}

template <int NQ, int MODE>
static tf_status launch(GatherParams p, int ug, cudaStream_t s) {
  const int per_sm = configure<NQ, MODE>();
  if (per_sm == 0) return TF_ERR_CUDA;
  // The window's few chunks per unit: at most 4 splits, merged inside one
  // cluster (timed at 128K with 32 units of one query head: 4 splits 5.55 us,
  // 8 splits 6.09 us per call); longer chunk lists keep more splits and the
  // ticketed merge.
  const int cap = MODE == kModeWindow ? (p.splits_cap < kWindowSplits ? p.splits_cap : kWindowSplits)
                                      : p.splits_cap;
  p.splits = wave_splits(ug, num_sms() * per_sm, cap);
  p.cmerge = (p.splits > 1 && p.splits <= kMaxClusterSplits) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, ug);
  cfg.blockDim = dim3(kGatherThreads);
  cfg.dynamicSmemBytes = kGatherSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.cmerge ? (unsigned)p.splits : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.cmerge ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, gather_attn_kernel<NQ, MODE>, p) != cudaSuccess) return TF_ERR_CUDA;
  return launch_status();
}

template <int NQ>
static tf_status launch_mode(int mode, const GatherParams& p, int ug, cudaStream_t s) {
  return mode == kModeChunks ? launch<NQ, kModeChunks>(p, ug, s) : launch<NQ, kModeWindow>(p, ug, s);
}

tf_status gather_launch(int mode, GatherParams p, int units, int rows, int P_max, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  if (p.T != 1) return TF_ERR_UNSUPPORTED;
  const int nq = gather_nq(rows);
  p.ngroups = (rows + nq - 1) / nq;
  p.splits_cap = gather_splits_cap(P_max);
  const int ug = units * p.ngroups;
  const size_t need = gather_workspace(units, rows, P_max);
  if (!ws || ws_bytes < need || !aligned16(ws)) return TF_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  p.tickets = reinterpret_cast<int*>(w);
  p.part_ml = reinterpret_cast<float*>(w + align_up((size_t)ug * sizeof(int), 256));
  p.part_o = reinterpret_cast<float*>(w + align_up((size_t)ug * sizeof(int), 256) +
                                      align_up((size_t)ug * p.splits_cap * nq * 2 * sizeof(float), 256));
  switch (nq) {
    case 1: return launch_mode<1>(mode, p, ug, stream);
    case 2: return launch_mode<2>(mode, p, ug, stream);
    default: return launch_mode<4>(mode, p, ug, stream);
  }
}

TF_DBG_READER(dbg_read_gather)

}  // namespace tf

// ------------------------------------------------------------------ C ABI

extern "C" size_t tf_sparse_decode_attn_workspace(int B, int Hq, int Hkv, int kc) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || kc <= 0 || Hq % Hkv) return 0;
  // the path tf_sparse_decode_attn takes for this head grouping
  return Hq / Hkv >= 2 ? tf::sparse_decode_umma_ws(B, Hq, Hkv, kc)
                       : tf::gather_workspace(B * Hkv, Hq / Hkv, kc * tf::kChunk);
}

extern "C" tf_status tf_sparse_decode_attn(const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                           const int32_t* seq_lens, const int32_t* idx, const int32_t* n_sel, int B,
                                           int Hq, int Hkv, int Lmax, int D, int chunk, int kc, float scale,
                                           float* out, void* ws, size_t ws_bytes, tf_stream_t stream) {
  using namespace tf;
  if (!q || !K || !V || !seq_lens || !idx || !n_sel || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || kc <= 0 || Hq % Hkv) return TF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  if (B == 0) return TF_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (Lmax == 0)  // no positions at all: every output row is zero
    return cudaMemsetAsync(out, 0, (size_t)B * Hq * kHeadDim * sizeof(float), st) == cudaSuccess ? TF_OK
                                                                                          : TF_ERR_CUDA;
  if (Hq / Hkv >= 2) {
    // GQA: the gathered verify kernel with one query token and no candidate
    // rows (8-row chunks land as 2 KB TMA boxes, QK^T and PV on tcgen05); the
    // group's heads share every key tile.  At 128K, batch 4 x 8 KV heads,
    // 4 heads each: 49.7 -> 30.9 us per call.  With one head per selection the
    // CUDA-core gather kernel below is faster (25.8 against 30.3 us).
    return sparse_decode_umma(q, K, V, seq_lens, idx, n_sel, B, Hq, Hkv, Lmax, kc, scale, out, ws, ws_bytes, st);
  }
  GatherParams p{};
  p.q = q; p.K = K; p.V = V; p.seq_lens = seq_lens; p.idx = idx; p.n_sel = n_sel;
  p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.T = 1; p.kc = kc;
  p.scale_log2 = scale * kLog2e; p.out = out;
  return gather_launch(kModeChunks, p, B * Hkv, Hq / Hkv, kc * kChunk, ws, ws_bytes, stream);
}

extern "C" size_t tf_stream_window_attn_workspace(int B, int Hq, int Hkv, int n_sink, int window) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || n_sink < 0 || window < 0 || Hq % Hkv) return 0;
  return tf::gather_workspace(B * Hkv, Hq / Hkv, n_sink + window);
}

extern "C" tf_status tf_stream_window_attn(const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                           const int32_t* seq_lens, int B, int Hq, int Hkv, int Lmax, int D,
                                           int n_sink, int window, float scale, float* out, void* ws,
                                           size_t ws_bytes, tf_stream_t stream) {
  using namespace tf;
  if (!q || !K || !V || !seq_lens || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || n_sink < 0 || window < 0 || Hq % Hkv) return TF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim) return TF_ERR_UNSUPPORTED;
  if (B == 0) return TF_OK;
  GatherParams p{};
  p.q = q; p.K = K; p.V = V; p.seq_lens = seq_lens;
  p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.T = 1;
  p.n_sink = n_sink; p.window = window;
  p.scale_log2 = scale * kLog2e; p.out = out;
  return gather_launch(kModeWindow, p, B * Hkv, Hq / Hkv, n_sink + window, ws, ws_bytes, stream);
}
