// a1 -- chunk-mean retrieval index for the Force 2 drafter.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": Force 2 retrieves KV blocks by key-query similarity; the page's
// "Production Advantages" section calls its bookkeeping an on-demand sparse
// index.  Here a block is 8 consecutive tokens represented by its mean key,
// rounded once to bf16 (nearest, ties to even).
//
// Design: a pure HBM stream.  One thread owns one 16-byte column slice (8 head
// dims) of one chunk: a chunk is 8 rows x 256 B = 2 KiB contiguous, so 16
// threads cover it and every load instruction of a half-warp reads 256
// contiguous bytes.  Each thread keeps all 8 row loads of its next item in
// flight while it sums the current one (the exact sums cost ~600 instructions
// per 128 bytes, so without the overlap the stream waits on the arithmetic).
// The sum of the rows is carried as an unevaluated fp32 pair (TwoSum), so the
// mean is exact before its single rounding to bf16.
#include "tf_common.cuh"

namespace tf {
namespace {

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Round the exact value hi + lo (|lo| <= ulp(hi)/2, both fp32) to bf16, nearest
// with ties to even.  The fp32 rounding of hi alone is right unless hi sits
// exactly on a bf16 midpoint; then the sign of lo decides, and only lo == 0 is a
// true tie.
__device__ __forceinline__ uint16_t round_pair_bf16(float hi, float lo) {
  uint32_t b = __float_as_uint(hi);
  if ((b & 0x7f800000u) == 0x7f800000u) return (uint16_t)((b >> 16) | ((b & 0xffffu) ? 0x40u : 0u));
  if ((b & 0xffffu) == 0x8000u && lo != 0.0f) {
    bool away = (lo > 0.0f) == (hi > 0.0f);
    return (uint16_t)((b >> 16) + (away ? 1u : 0u));
  }
  uint32_t lsb = (b >> 16) & 1u;
  return (uint16_t)((b + 0x7fffu + lsb) >> 16);
}

// One item = (unit, chunk, 16-byte column slice): where its rows start and how
// many of them the sequence holds.
struct Item {
  const uint16_t* src;
  uint16_t* dst;
  int n;
  bool ok;  // (debug builds) the chunk lies inside the index and its rows inside the cache
};

// A thread's walk over the items.  The grid stride is a multiple of 16 items,
// so a thread keeps its column slice and steps through (b, g, c) by a fixed
// (db, dg, dc) with carries: no integer division per item.
struct Walk {
  int b, g, c;     // sequence, KV head, chunk (from c_begin)
  int db, dg, dc;  // the step per grid stride
  int slice;
};

__device__ __forceinline__ Item item_at(const Walk& w, const uint16_t* K, const int32_t* seq_lens, int Hkv,
                                        int Lmax, int Cmax, int c_begin, uint16_t* M) {
  const int c = c_begin + w.c;
  const size_t bg = (size_t)w.b * Hkv + w.g;
  const int L = clamp_len(seq_lens[w.b], Lmax);
  int n = L - c * kChunk;
  n = n < 0 ? 0 : (n > kChunk ? kChunk : n);
  Item it;
  it.src = K + (bg * Lmax + (size_t)c * kChunk) * kHeadDim + w.slice * 8;
  it.dst = M + (bg * Cmax + c) * kHeadDim + w.slice * 8;
  it.ok = TF_DBG_OK(c >= 0 && c < Cmax, kDbgIndexRow) && TF_DBG_OK(n == 0 || c * kChunk + n <= L, kDbgCacheRow);
  it.n = it.ok ? n : 0;
  return it;
}

__device__ __forceinline__ void advance(Walk& w, int Hkv, int n_chunks) {
  w.c += w.dc;
  int carry = 0;
  if (w.c >= n_chunks) {
    w.c -= n_chunks;
    carry = 1;
  }
  w.g += w.dg + carry;  // < 2 Hkv
  w.b += w.db;
  if (w.g >= Hkv) {
    w.g -= Hkv;
    w.b += 1;
  }
}

__device__ __forceinline__ void load_rows(const Item& it, uint4 (&rows)[kChunk]) {
#pragma unroll
  for (int r = 0; r < kChunk; ++r)
    rows[r] = (r < it.n) ? ld_stream16(it.src + (size_t)r * kHeadDim) : make_uint4(0, 0, 0, 0);
}

// Exact mean of the rows, rounded once to bf16, stored as 8 head dims.
__device__ __forceinline__ void mean_store(const Item& it, const uint4 (&rows)[kChunk]) {
  if (!it.ok) return;
  float hi[8], lo[8];
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    hi[d] = 0.0f;
    lo[d] = 0.0f;
  }
#pragma unroll
  for (int r = 0; r < kChunk; ++r) {
    float f[8];
    unpack8(rows[r], f);
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      float s, e;
      two_sum(hi[d], f[d], s, e);
      hi[d] = s;
      lo[d] += e;
    }
  }
  const int n = it.n;
  uint32_t packed[4];
#pragma unroll
  for (int d = 0; d < 8; d += 2) {
    uint16_t o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float h = hi[d + k], l = lo[d + k];
      float s, e;
      two_sum(h, l, s, e);  // renormalise the pair
      h = s;
      l = e;
      if (n == 0) {
        o[k] = 0;
      } else if (n == kChunk) {
        o[k] = round_pair_bf16(h * 0.125f, l * 0.125f);  // exact scaling by 2^-3
      } else {
        // Pair divided by n: quotient, exact remainder by FMA, corrected low part.
        const float fn = (float)n;
        float qh = __fdiv_rn(h, fn);
        float rem = fmaf(-qh, fn, h);
        float ql = __fdiv_rn(rem + l, fn);
        float s2, e2;
        two_sum(qh, ql, s2, e2);
        o[k] = round_pair_bf16(s2, e2);
      }
    }
    packed[d / 2] = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
  }
  *reinterpret_cast<uint4*>(it.dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// Grid-stride over items, software-pipelined: the next item's eight row loads
// are issued before the current item's sums, so the DRAM round trip overlaps
// the arithmetic.
__global__ void __launch_bounds__(256) chunk_means_kernel(const uint16_t* __restrict__ K,
                                                          const int32_t* __restrict__ seq_lens, int B,
                                                          int Hkv, int Lmax, int c_begin, int n_chunks,
                                                          uint16_t* __restrict__ M) {
  const int Cmax = (Lmax + kChunk - 1) / kChunk;
  pdl_wait();
  const long long item0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long step = (long long)gridDim.x * blockDim.x / 16;  // chunks per grid stride
  const long long ci = item0 / 16;
  Walk w;
  w.slice = (int)(item0 % 16);
  w.c = (int)(ci % n_chunks);
  w.g = (int)(ci / n_chunks % Hkv);
  const long long b0 = ci / n_chunks / Hkv;
  if (b0 >= B) return;
  w.b = (int)b0;
  w.dc = (int)(step % n_chunks);
  w.dg = (int)(step / n_chunks % Hkv);
  w.db = (int)(step / n_chunks / Hkv);
  Item cur = item_at(w, K, seq_lens, Hkv, Lmax, Cmax, c_begin, M);
  uint4 rows[kChunk];
  load_rows(cur, rows);
  while (true) {
    advance(w, Hkv, n_chunks);
    const bool more = w.b < B;
    Item nxt = cur;
    uint4 next_rows[kChunk];
    if (more) {
      nxt = item_at(w, K, seq_lens, Hkv, Lmax, Cmax, c_begin, M);
      load_rows(nxt, next_rows);
    }
    mean_store(cur, rows);
    if (!more) break;
#pragma unroll
    for (int r = 0; r < kChunk; ++r) rows[r] = next_rows[r];
    cur = nxt;
  }
}

}  // namespace

TF_DBG_READER(dbg_read_chunk_means)

}  // namespace tf

extern "C" tf_status tf_build_chunk_means(const uint16_t* K, const int32_t* seq_lens, int B, int Hkv,
                                          int Lmax, int D, int chunk, int c_begin, int c_end, uint16_t* M,
                                          tf_stream_t stream) {
  using namespace tf;
  if (!K || !seq_lens || !M || B < 0 || Hkv < 0 || Lmax < 0) return TF_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(M)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;
  if (c_begin < 0 || c_end < c_begin || c_end > Cmax) return TF_ERR_INVALID_ARG;
  const int n_chunks = c_end - c_begin;
  const long long total = (long long)B * Hkv * n_chunks * 16;
  if (total == 0) return TF_OK;
  constexpr int threads = 256;
  static_assert(threads % 16 == 0, "the grid stride must keep each thread's column slice");
  long long blocks = (total + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (launch_pdl(chunk_means_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, K, seq_lens, B, Hkv, Lmax,
                 c_begin, n_chunks, M) != cudaSuccess)
    return TF_ERR_CUDA;
  return launch_status();
}
