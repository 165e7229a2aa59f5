// Library-wide entry points of the C ABI: status strings, version and the
// device-side status of a workspace.
#include "tf_common.cuh"

extern "C" const char* tf_status_string(tf_status s) {
  switch (s) {
    case TF_OK: return "ok";
    case TF_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, inconsistent sizes)";
    case TF_ERR_UNSUPPORTED: return "unsupported shape (head dim must be 128, chunk must be 8)";
    case TF_ERR_WORKSPACE: return "workspace missing, misaligned or smaller than the *_workspace() size";
    case TF_ERR_CUDA: return "CUDA launch failed";
    case TF_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the static buffer of the no-allocation entry point";
    case TF_ERR_DEVICE_DATA: return "a kernel flagged an error on the device; the outputs since the last check are invalid";
  }
  return "unknown status";
}

extern "C" int tf_abi_version(void) { return 101; }

extern "C" tf_status tf_check_status(void* ws, size_t ws_bytes, tf_stream_t stream) {
  if (!ws || ws_bytes < sizeof(int32_t)) return TF_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return TF_ERR_CUDA;
  if (word == 0) return TF_OK;
  if (cudaMemsetAsync(ws, 0, ws_bytes, s) != cudaSuccess) return TF_ERR_CUDA;
  return TF_ERR_DEVICE_DATA;
}

extern "C" tf_status tf_debug_status(uint32_t* flags, int clear) {
  if (!flags) return TF_ERR_INVALID_ARG;
  *flags = 0;
#ifdef TF_DEBUG
  using namespace tf;
  const uint32_t words[] = {dbg_read_chunk_means(clear), dbg_read_gather(clear), dbg_read_verify(clear),
                            dbg_read_topk(clear),        dbg_read_draft(clear),  dbg_read_pack(clear)};
  for (uint32_t w : words) {
    if (w == ~0u) return TF_ERR_CUDA;
    *flags |= w;
  }
  return TF_OK;
#else
  (void)clear;
  return TF_ERR_UNSUPPORTED;
#endif
}
