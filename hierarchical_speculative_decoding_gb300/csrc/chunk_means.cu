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
// mean is exact before its single rounding to bf16.  Columns whose pair is not
// finite (infinities or NaNs among the keys, or sums beyond the fp32 range)
// are redone after the stream with the inputs scaled by 1/8 first.
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

// Exact mean of the n rows at src (pairs of fp32 by TwoSum), rounded once to
// bf16 and stored at dst.  Out of line and reading its rows again itself, so
// the rare call leaves the streaming loop's code as it is.
// Every input is first scaled by 2^-3, which is exact for every bf16 value (its
// smallest subnormal, 2^-133, stays an fp32 subnormal), so no partial sum can
// overflow however large the keys.  A column holding an infinity or a NaN
// takes the IEEE sum's outcome: +-inf, or NaN (0x7fc0) for a NaN or opposite
// infinities.
__device__ __noinline__ void exact_means(const uint16_t* __restrict__ src, int n, uint16_t* __restrict__ dst) {
  uint4 rows[kChunk];
#pragma unroll
  for (int r = 0; r < kChunk; ++r)
    rows[r] = (r < n) ? *reinterpret_cast<const uint4*>(src + (size_t)r * kHeadDim) : make_uint4(0, 0, 0, 0);
  uint16_t o[8];
  float hi[8], lo[8], plain[8];
  bool special[8];
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    hi[d] = 0.0f;
    lo[d] = 0.0f;
    plain[d] = 0.0f;
    special[d] = false;
  }
#pragma unroll
  for (int r = 0; r < kChunk; ++r) {
    float f[8];
    unpack8(rows[r], f);
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      const float x = f[d] * 0.125f;
      special[d] |= !isfinite(f[d]);
      plain[d] += x;
      float s, e;
      two_sum(hi[d], x, s, e);
      hi[d] = s;
      lo[d] += e;
    }
  }
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    float h = hi[d], l = lo[d];
    float s, e;
    two_sum(h, l, s, e);  // renormalise the pair
    h = s;
    l = e;
    if (n == 0) {
      o[d] = 0;
    } else if (special[d]) {
      o[d] = isnan(plain[d]) ? (uint16_t)0x7fc0u : (plain[d] > 0.0f ? (uint16_t)0x7f80u : (uint16_t)0xff80u);
    } else if (n == kChunk) {
      o[d] = round_pair_bf16(h, l);  // the scaled sum is the mean
    } else {
      // Pair divided by n / 8: quotient, exact remainder by FMA, corrected low part.
      const float fn = (float)n * 0.125f;
      float qh = __fdiv_rn(h, fn);
      float rem = fmaf(-qh, fn, h);
      float ql = __fdiv_rn(rem + l, fn);
      float s2, e2;
      two_sum(qh, ql, s2, e2);
      o[d] = round_pair_bf16(s2, e2);
    }
  }
  uint32_t packed[4];
#pragma unroll
  for (int d = 0; d < 8; d += 2) packed[d / 2] = (uint32_t)o[d] | ((uint32_t)o[d + 1] << 16);
  *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// Exact mean of the rows, rounded once to bf16, stored as 8 head dims: the sum
// of the rows carried as an unevaluated fp32 pair (TwoSum), renormalised,
// scaled by 1/8 (or divided by the row count of a partial chunk) and rounded
// once.  A column whose pair is not finite -- an infinity or NaN among the
// keys, or partial sums beyond the fp32 range -- returns false; the item is
// redone after the stream with inputs scaled by 1/8 first and IEEE results
// for infinities and NaNs.
__device__ __forceinline__ bool mean_store(const Item& it, const uint4 (&rows)[kChunk]) {
  if (!it.ok) return true;
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
  uint16_t o[8];
  bool finite = true;
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    float h = hi[d], l = lo[d];
    float s, e;
    two_sum(h, l, s, e);  // renormalise the pair
    h = s;
    l = e;
    finite &= isfinite(h) && isfinite(l);
    if (n == 0) {
      o[d] = 0;
    } else if (n == kChunk) {
      o[d] = round_pair_bf16(h * 0.125f, l * 0.125f);  // exact scaling by 2^-3
    } else {
      // Pair divided by n: quotient, exact remainder by FMA, corrected low part.
      const float fn = (float)n;
      float qh = __fdiv_rn(h, fn);
      float rem = fmaf(-qh, fn, h);
      float ql = __fdiv_rn(rem + l, fn);
      float s2, e2;
      two_sum(qh, ql, s2, e2);
      o[d] = round_pair_bf16(s2, e2);
    }
  }
  if (!finite) return false;  // redone after the stream
  uint32_t packed[4];
#pragma unroll
  for (int d = 0; d < 8; d += 2) packed[d / 2] = (uint32_t)o[d] | ((uint32_t)o[d + 1] << 16);
  *reinterpret_cast<uint4*>(it.dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  return true;
}

// Items of one thread whose means are redone exactly after its stream, by
// their step number in the thread's walk: four slots in registers (constant
// indices only); more than four (only keys built to sit on rounding midpoints)
// redo the thread's whole walk.
struct Deferred {
  int step[4];
  int count;
  __device__ __forceinline__ void add(int k) {
    switch (count) {
      case 0: step[0] = k; break;
      case 1: step[1] = k; break;
      case 2: step[2] = k; break;
      case 3: step[3] = k; break;
      default: break;
    }
    ++count;
  }
};

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
  const Walk w0 = w;
  Deferred later;
  later.count = 0;
  int k = 0;  // step of the walk
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
    if (!mean_store(cur, rows)) later.add(k);
    if (!more) break;
#pragma unroll
    for (int r = 0; r < kChunk; ++r) rows[r] = next_rows[r];
    cur = nxt;
    ++k;
  }
  if (later.count == 0) return;
  // the deferred steps, in increasing order, by walking again
  int j = 0;
  w = w0;
  for (int kk = 0; w.b < B; ++kk, advance(w, Hkv, n_chunks)) {
    bool redo = later.count > 4;
#pragma unroll
    for (int t = 0; t < 4; ++t) redo |= t < later.count && later.step[t] == kk;
    if (!redo) continue;
    const Item it = item_at(w, K, seq_lens, Hkv, Lmax, Cmax, c_begin, M);
    if (it.ok && it.n > 0) exact_means(it.src, it.n, it.dst);
    if (later.count <= 4 && ++j == later.count) break;
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
