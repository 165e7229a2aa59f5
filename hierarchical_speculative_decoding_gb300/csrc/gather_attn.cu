// a4, a6 (+ a5) -- decode attention over a gathered set of KV positions.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce":
//   Force 2 (retrieval drafter): the target model attends only to the KV
//     blocks retrieved by key-query similarity (the selected chunk list);
//   Force 1 (streaming drafter): attention sinks plus the most recent window.
// Both are one query token per head attending to a small, irregular subset of
// a long cache, so both run through one kernel parameterised by how a
// "virtual row" (the i-th position of the set) maps to a cache position.
//
// Design (HBM-bound, ~1 flop/byte): split-K over the position set.  Each warp
// walks groups of 8 virtual rows; a half-warp owns a row and each lane reads 16
// bytes (8 head dims) of K and of V with L1-bypassing vector loads, so one
// load instruction moves 2 x 256 contiguous bytes and each lane keeps 8 loads
// in flight.  Scores are reduced over the half-warp with 4 shuffles, the
// online softmax runs in the log2 domain in fp32, warps merge in shared
// memory, and splits merge with the log-sum-exp identity in the last CTA of
// each unit to finish (atomic ticket, no waiting).
#include "gather_attn.cuh"

namespace tf {

template <int NQ, int MODE>
__global__ void __launch_bounds__(kGatherThreads) gather_attn_kernel(GatherParams p) {
  constexpr int kW = kGatherThreads / 32;
  __shared__ float sm_m[kW][NQ], sm_l[kW][NQ];
  __shared__ float sm_o[kW][NQ][kHeadDim];
  __shared__ int s_last;

  const int unit_grp = blockIdx.y;
  const int unit = unit_grp / p.ngroups, grp = unit_grp % p.ngroups;
  const int b = unit / p.Hkv, g = unit % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int rows = G * p.T;
  const int L = clamp_len(p.seq_lens[b], p.Lmax);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane >> 4, l16 = lane & 15;

  // ---- the position set of this unit
  int P = 0, ns_eff = 0, w0 = 0, nsel = 0;
  const int32_t* sel = nullptr;
  if (MODE == kModeChunks) {
    nsel = p.n_sel[unit];
    nsel = nsel < 0 ? 0 : (nsel > p.kc ? p.kc : nsel);
    sel = p.idx + (size_t)unit * p.kc;
    P = nsel * kChunk;
  } else {
    ns_eff = min(p.n_sink, L);
    w0 = max(p.n_sink, L - p.window);
    P = ns_eff + max(0, L - w0);
  }
  const int C = (L + kChunk - 1) / kChunk;

  // ---- this CTA's query rows: r = hh * T + j, head h = g * G + hh
  float qv[NQ][8];
  int lim[NQ];
  bool row_on[NQ];
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    const int rr = grp * NQ + r;
    row_on[r] = rr < rows;
    const int hh = row_on[r] ? rr / p.T : 0, j = row_on[r] ? rr % p.T : 0;
    lim[r] = row_on[r] ? 0x7fffffff : -1;
    const uint16_t* qrow = p.q + (((size_t)b * p.Hq + (size_t)g * G + hh) * p.T + j) * kHeadDim + l16 * 8;
    float f[8];
    unpack8(row_on[r] ? *reinterpret_cast<const uint4*>(qrow) : make_uint4(0, 0, 0, 0), f);
#pragma unroll
    for (int d = 0; d < 8; ++d) qv[r][d] = f[d] * p.scale_log2;
  }

  // ---- split range over virtual rows (whole groups of 8)
  int vper = (P + p.splits - 1) / p.splits;
  vper = (vper + 7) & ~7;
  const int v_begin = blockIdx.x * vper;
  const int v_end = min(P, v_begin + vper);

  float m[NQ], l[NQ], o[NQ][8];
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int d = 0; d < 8; ++d) o[r][d] = 0.0f;
  }

  const size_t kv_base = (size_t)unit * p.Lmax;
  for (int gv = v_begin + warp * 8; gv < v_end; gv += kW * 8) {
    uint4 kr[4], vr[4];
    int pos[4];
    bool ok[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = gv + sub + 2 * i;
      int t = -1;
      if (v < v_end) {
        if (MODE == kModeChunks) {
          const int c = sel[v >> 3];
          t = (c >= 0 && c < C) ? c * kChunk + (v & 7) : -1;
          if (t >= L) t = -1;
        } else {
          t = (v < ns_eff) ? v : w0 + (v - ns_eff);
        }
      }
      pos[i] = t;
      ok[i] = t >= 0;
      const size_t off = (kv_base + (size_t)(ok[i] ? t : 0)) * kHeadDim + l16 * 8;
      kr[i] = ok[i] ? ld_stream16(p.K + off) : make_uint4(0, 0, 0, 0);
      vr[i] = ok[i] ? ld_stream16(p.V + off) : make_uint4(0, 0, 0, 0);
    }
    float s[4][NQ];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float kf[8];
      unpack8(kr[i], kf);
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        float a = 0.0f;
#pragma unroll
        for (int d = 0; d < 8; ++d) a = fmaf(qv[r][d], kf[d], a);
        a += __shfl_xor_sync(0xffffffffu, a, 8);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        s[i][r] = (ok[i] && pos[i] <= lim[r]) ? a : -INFINITY;
      }
    }
    float vf[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack8(vr[i], vf[i]);
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      const float mx = fmaxf(fmaxf(s[0][r], s[1][r]), fmaxf(s[2][r], s[3][r]));
      const float mn = fmaxf(m[r], mx);
      if (mn == -INFINITY) continue;
      const float alpha = merge_scale(m[r], mn);
      float pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = exp2f(s[i][r] - mn);
      l[r] = l[r] * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        float acc = o[r][d] * alpha;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc = fmaf(pr[i], vf[i][d], acc);
        o[r][d] = acc;
      }
      m[r] = mn;
    }
  }

  // ---- merge the two half-warps (different rows, same query rows)
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m[r], 16);
    const float l2 = __shfl_xor_sync(0xffffffffu, l[r], 16);
    const float mn = fmaxf(m[r], m2);
    const float a1 = merge_scale(m[r], mn), a2 = merge_scale(m2, mn);
    l[r] = l[r] * a1 + l2 * a2;
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      const float o2 = __shfl_xor_sync(0xffffffffu, o[r][d], 16);
      o[r][d] = o[r][d] * a1 + o2 * a2;
    }
    m[r] = mn;
  }
  if (sub == 0) {
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      if (l16 == 0) {
        sm_m[warp][r] = m[r];
        sm_l[warp][r] = l[r];
      }
#pragma unroll
      for (int d = 0; d < 8; ++d) sm_o[warp][r][l16 * 8 + d] = o[r][d];
    }
  }
  __syncthreads();

  // ---- merge warps: thread handles (r, d) pairs
  const int out_rows = min(NQ, rows - grp * NQ);
  float* part_ml = p.part_ml + ((size_t)unit_grp * p.splits_cap + blockIdx.x) * NQ * 2;
  float* part_o = p.part_o + ((size_t)unit_grp * p.splits_cap + blockIdx.x) * NQ * kHeadDim;
  for (int pr = threadIdx.x; pr < out_rows * kHeadDim; pr += kGatherThreads) {
    const int r = pr / kHeadDim, d = pr % kHeadDim;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW; ++w) mx = fmaxf(mx, sm_m[w][r]);
    float ls = 0.0f, os = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const float f = merge_scale(sm_m[w][r], mx);
      ls = fmaf(f, sm_l[w][r], ls);
      os = fmaf(f, sm_o[w][r][d], os);
    }
    if (p.splits == 1) {
      const int rr = grp * NQ + r;
      const int hh = rr / p.T, j = rr % p.T;
      p.out[(((size_t)b * p.Hq + (size_t)g * G + hh) * p.T + j) * kHeadDim + d] = (ls > 0.0f) ? os / ls : 0.0f;
    } else {
      if (d == 0) {
        part_ml[r * 2 + 0] = mx;
        part_ml[r * 2 + 1] = ls;
      }
      part_o[r * kHeadDim + d] = os;
    }
  }
  if (p.splits == 1) return;

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&p.tickets[unit_grp], 1) == p.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const float* ml0 = p.part_ml + (size_t)unit_grp * p.splits_cap * NQ * 2;
  const float* o0 = p.part_o + (size_t)unit_grp * p.splits_cap * NQ * kHeadDim;
  for (int pr = threadIdx.x; pr < out_rows * kHeadDim; pr += kGatherThreads) {
    const int r = pr / kHeadDim, d = pr % kHeadDim;
    float mx = -INFINITY;
    for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, __ldcg(ml0 + ((size_t)s * NQ + r) * 2));
    float ls = 0.0f, os = 0.0f;
    for (int s = 0; s < p.splits; ++s) {
      const float f = merge_scale(__ldcg(ml0 + ((size_t)s * NQ + r) * 2), mx);
      ls = fmaf(f, __ldcg(ml0 + ((size_t)s * NQ + r) * 2 + 1), ls);
      os = fmaf(f, __ldcg(o0 + ((size_t)s * NQ + r) * kHeadDim + d), os);
    }
    const int rr = grp * NQ + r;
    const int hh = rr / p.T, j = rr % p.T;
    p.out[(((size_t)b * p.Hq + (size_t)g * G + hh) * p.T + j) * kHeadDim + d] = (ls > 0.0f) ? os / ls : 0.0f;
  }
  if (threadIdx.x == 0) p.tickets[unit_grp] = 0;
}

// ------------------------------------------------------------------ host side

int gather_nq(int rows) {
  if (rows <= 1) return 1;
  if (rows <= 2) return 2;
  if (rows <= 4) return 4;
  if (rows <= 6) return 6;
  return 8;
}

int gather_splits_cap(int P_max) {
  int s = (P_max + 63) / 64;
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

template <int NQ>
static void launch_nq(int mode, const GatherParams& p, dim3 grid, cudaStream_t s) {
  switch (mode) {
    case kModeChunks: gather_attn_kernel<NQ, kModeChunks><<<grid, kGatherThreads, 0, s>>>(p); break;
    default: gather_attn_kernel<NQ, kModeWindow><<<grid, kGatherThreads, 0, s>>>(p); break;
  }
}

tf_status gather_launch(int mode, GatherParams p, int units, int rows, int P_max, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  const int nq = gather_nq(rows);
  p.ngroups = (rows + nq - 1) / nq;
  p.splits_cap = gather_splits_cap(P_max);
  const int ug = units * p.ngroups;
  const int target = num_sms() * 4;
  int splits = (target + ug - 1) / ug;
  if (splits > p.splits_cap) splits = p.splits_cap;
  p.splits = splits < 1 ? 1 : splits;
  const size_t need = gather_workspace(units, rows, P_max);
  if (p.splits > 1 && (!ws || ws_bytes < need || !aligned16(ws))) return TF_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  p.tickets = reinterpret_cast<int*>(w);
  p.part_ml = reinterpret_cast<float*>(w + align_up((size_t)ug * sizeof(int), 256));
  p.part_o = reinterpret_cast<float*>(w + align_up((size_t)ug * sizeof(int), 256) +
                                      align_up((size_t)ug * p.splits_cap * nq * 2 * sizeof(float), 256));
  dim3 grid(p.splits, ug);
  switch (nq) {
    case 1: launch_nq<1>(mode, p, grid, stream); break;
    case 2: launch_nq<2>(mode, p, grid, stream); break;
    case 4: launch_nq<4>(mode, p, grid, stream); break;
    case 6: launch_nq<6>(mode, p, grid, stream); break;
    default: launch_nq<8>(mode, p, grid, stream); break;
  }
  return launch_status();
}

}  // namespace tf

// ------------------------------------------------------------------ C ABI

extern "C" size_t tf_sparse_decode_attn_workspace(int B, int Hq, int Hkv, int kc) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || kc <= 0 || Hq % Hkv) return 0;
  return tf::gather_workspace(B * Hkv, Hq / Hkv, kc * tf::kChunk);
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
