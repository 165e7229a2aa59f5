// a7 (+ a5) -- full-cache verification attention (Force 3).
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": the target model with the complete KV cache checks all drafted
// candidates in one parallel pass.  The candidates form a chain whose keys
// already sit at positions L-T .. L-1, so query j sees positions [0, L-T+j].
#include "gather_attn.cuh"

extern "C" size_t tf_verify_attn_workspace(int B, int Hq, int Hkv, int Lmax, int T) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lmax <= 0 || T <= 0 || Hq % Hkv) return 0;
  return tf::gather_workspace(B * Hkv, (Hq / Hkv) * T, Lmax);
}

extern "C" tf_status tf_verify_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                                    const int32_t* seq_lens, int B, int Hq, int Hkv, int Lmax, int D, int T,
                                    float scale, float* out, void* ws, size_t ws_bytes, tf_stream_t stream) {
  using namespace tf;
  if (!Q || !K || !V || !seq_lens || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || Hq % Hkv || T < 1) return TF_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || T > 16) return TF_ERR_UNSUPPORTED;
  if (B == 0) return TF_OK;
  GatherParams p{};
  p.q = Q; p.K = K; p.V = V; p.seq_lens = seq_lens;
  p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.T = T;
  p.scale_log2 = scale * kLog2e; p.out = out;
  return gather_launch(kModePrefix, p, B * Hkv, (Hq / Hkv) * T, Lmax, ws, ws_bytes, stream);
}
