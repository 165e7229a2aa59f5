// Library-wide entry points of the C ABI: status strings and version.
#include "tf_common.cuh"

extern "C" const char* tf_status_string(tf_status s) {
  switch (s) {
    case TF_OK: return "ok";
    case TF_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, inconsistent sizes)";
    case TF_ERR_UNSUPPORTED: return "unsupported shape (head dim must be 128, chunk must be 8)";
    case TF_ERR_WORKSPACE: return "workspace missing, misaligned or smaller than the *_workspace() size";
    case TF_ERR_CUDA: return "CUDA launch failed";
    case TF_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the static buffer of the no-allocation entry point";
  }
  return "unknown status";
}

extern "C" int tf_abi_version(void) { return 100; }
