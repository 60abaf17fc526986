// Library-wide entry points of libvt: status text and ABI version.
#include "vt_common.cuh"

extern "C" const char* vt_status_string(int status) {
  switch (status) {
    case VT_OK: return "ok";
    case VT_ERR_INVALID_ARG: return "invalid argument";
    case VT_ERR_UNSUPPORTED: return "unsupported";
    case VT_ERR_CUDA: return "CUDA error";
    case VT_ERR_BAD_INPUT: return "bad input data";
    case VT_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case VT_ERR_SCRATCH_LIMIT: return "problem exceeds the library's static scratch";
    default: return "unknown status";
  }
}

extern "C" int vt_abi_version(void) { return 100; }
