// tf_sparse_decode_attn_noalloc -- the retrieval-sparse decode attention of
// tf_sparse_decode_attn for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: plugins hosted by an inference
// engine that owns every device allocation and hands out only the tensors of a
// call, or latency-critical loops where an allocation (and the implicit device
// synchronisation it can bring) is not allowed.  This entry point takes the
// same inputs and outputs as tf_sparse_decode_attn but no workspace: its
// split-K scratch lives in one file-scope device array of a fixed size (32 MiB)
// that every GPU loading this library keeps until the process exits.  It always
// runs the CUDA-core gather kernel, also for grouped-query heads, where the
// workspace entry point runs the tensor-core kernel: the two agree within the
// attention tolerance (2e-3), not bit for bit.
//
// Set-up happens on the first successful call made on each device (with that
// device current): the array's device address is looked up with
// cudaGetSymbolAddress and its ticket area is zeroed with a synchronous
// cudaMemset.  That first call therefore must come before any stream capture;
// made on a stream that is being captured it is refused (TF_ERR_INVALID_ARG)
// without touching the device, and a set-up that failed is tried again by the
// next call.  Every call shares the array and leaves its last contents behind;
// the tickets are reset by each call, the partial results are always rewritten
// before they are read.  Calls that overlap on the GPU (different streams, no
// ordering) race on the array.
#include <mutex>

#include "gather_attn.cuh"

namespace tf {
namespace {

constexpr size_t kScratchBytes = 32u << 20;  // 32 MiB per device
constexpr size_t kTicketArea = 64u << 10;    // tickets live in the first 64 KiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_sparse_scratch[kScratchBytes];

struct DeviceScratch {
  std::mutex mu;
  void* ptr = nullptr;  // set once the set-up succeeded
};
DeviceScratch g_dev[kMaxDevices];

// Device address of the scratch array on the current device.  The set-up runs
// under a per-device lock until it succeeds once; a failed attempt leaves
// nothing behind, so a later call tries again.  A stream under capture is
// refused before the device is touched (the synchronous set-up would end the
// capture).
void* scratch_for_current_device(cudaStream_t stream, tf_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *st = TF_ERR_CUDA;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *st = TF_ERR_UNSUPPORTED;
    return nullptr;
  }
  DeviceScratch& d = g_dev[dev];
  std::lock_guard<std::mutex> lock(d.mu);
  if (!d.ptr) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
      (void)cudaGetLastError();
      *st = TF_ERR_CUDA;
      return nullptr;
    }
    if (cap != cudaStreamCaptureStatusNone) {
      *st = TF_ERR_INVALID_ARG;
      return nullptr;
    }
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_sparse_scratch);
    if (e == cudaSuccess) e = cudaMemset(p, 0, kTicketArea);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      *st = TF_ERR_CUDA;
      return nullptr;
    }
    d.ptr = p;
  }
  *st = TF_OK;
  return d.ptr;
}

}  // namespace
}  // namespace tf

extern "C" tf_status tf_sparse_decode_attn_noalloc(const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                                   const int32_t* seq_lens, const int32_t* idx,
                                                   const int32_t* n_sel, int B, int Hq, int Hkv, int Lmax, int D,
                                                   int chunk, int kc, float scale, float* out,
                                                   tf_stream_t stream) {
  using namespace tf;
  if (!q || !K || !V || !seq_lens || !idx || !n_sel || !out) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || kc <= 0 || Hq % Hkv) return TF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  if (B == 0) return TF_OK;

  // The same layout the workspace path uses: tickets, then partial results.
  // Placed so the tickets always end at kTicketArea and the partials always
  // start there: a later, larger call never finds stale partials in its tickets.
  const int units = B * Hkv, rows = Hq / Hkv;
  const size_t need = gather_workspace(units, rows, kc * kChunk);
  const int nq = gather_nq(rows);
  const size_t ug = (size_t)units * ((rows + nq - 1) / nq);
  const size_t tickets = align_up(ug * sizeof(int), 256);
  if (tickets > kTicketArea || need - tickets > kScratchBytes - kTicketArea) return TF_ERR_SCRATCH_LIMIT;

  tf_status st;
  char* base = static_cast<char*>(scratch_for_current_device((cudaStream_t)stream, &st));
  if (!base) return st;
  char* ws = base + (kTicketArea - tickets);
  GatherParams p{};
  p.q = q; p.K = K; p.V = V; p.seq_lens = seq_lens; p.idx = idx; p.n_sel = n_sel;
  p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.T = 1; p.kc = kc;
  p.scale_log2 = scale * kLog2e; p.out = out;
  return gather_launch(kModeChunks, p, units, rows, kc * kChunk, ws, kScratchBytes - (kTicketArea - tickets),
                       stream);
}
