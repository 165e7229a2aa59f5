// Decode attention over a gathered position set (sparse chunks or sink +
// window); shared by the sparse and window entry points.
#pragma once

#include "tf_common.cuh"

namespace tf {

constexpr int kGatherThreads = 160;  // 4 compute warps + 1 bulk-copy producer warp
constexpr int kModeChunks = 0;  // positions of the selected chunks (Force 2)
constexpr int kModeWindow = 1;  // attention sinks + recent window (Force 1)

struct GatherParams {
  const uint16_t* q;  // [B, Hq, T, D]
  const uint16_t* K;  // [B, Hkv, Lmax, D]
  const uint16_t* V;
  const int32_t* seq_lens;
  const int32_t* idx;    // [B, Hkv, kc] (chunks mode)
  const int32_t* n_sel;  // [B, Hkv]     (chunks mode)
  int Hq, Hkv, Lmax, T, kc, n_sink, window;
  float scale_log2;  // softmax scale * log2(e)
  int ngroups;       // query-head groups per unit (<= 4 heads each)
  int splits;        // CTAs per (unit, group)
  int splits_cap;    // partial-buffer stride
  float* out;        // [B, Hq, T, D]
  int* tickets;      // [units * ngroups]
  float* part_ml;    // [units * ngroups, splits_cap, NQ, 2]
  float* part_o;     // [units * ngroups, splits_cap, NQ, D]
  int cmerge;        // 1: the splits of a (unit, group) form a cluster and merge through DSMEM
};

// The retrieval drafter's decode attention on the tensor cores: the gathered
// verify kernel (verify_attn.cu) with one query token per head and no
// candidate rows.  Arguments validated by the caller.
size_t sparse_decode_umma_ws(int B, int Hq, int Hkv, int kc);
tf_status sparse_decode_umma(const uint16_t* q, const uint16_t* K, const uint16_t* V, const int32_t* seq_lens,
                             const int32_t* idx, const int32_t* n_sel, int B, int Hq, int Hkv, int Lmax, int kc,
                             float scale, float* out, void* ws, size_t ws_bytes, cudaStream_t stream);

int gather_nq(int rows);  // query rows per CTA for `rows` rows per unit
size_t gather_workspace(int units, int rows, int P_max);
tf_status gather_launch(int mode, GatherParams p, int units, int rows, int P_max, void* ws, size_t ws_bytes,
                        cudaStream_t stream);

}  // namespace tf
