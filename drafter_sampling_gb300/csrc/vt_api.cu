// Library-wide entry points of libvt: status text, ABI version and the
// self-test of the bounded waits.
#include "vt_common.cuh"
#include "vt_umma.cuh"

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

namespace vt {
namespace {

constexpr uint32_t kSelftestMaxLimit = 1u << 20;

// One thread runs one bounded wait of the library on an object that nothing
// completes (or, for the control, one already complete) and records
// VT_DEV_TIMEOUT when the wait gives up.
__global__ void selftest_wait_kernel(int which, uint32_t limit, const unsigned* flag,
                                     int* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  bool done;
  if (which == 2) {
    done = (poll_published(flag, ld_relaxed_u32(flag), limit) >> 31) != 0u;
  } else {
    umma::mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (which == 1) umma::mbar_arrive(&bar);
    done = umma::mbar_wait(&bar, 0, limit);
  }
  if (!done) atomicOr(dev_status, VT_DEV_TIMEOUT);
}

}  // namespace
}  // namespace vt

extern "C" int vt_selftest_wait(int32_t which, uint32_t limit, const uint32_t* flag,
                                int32_t* dev_status, void* stream) {
  if (which < 0 || which > 2 || limit < 1 || limit > vt::kSelftestMaxLimit ||
      dev_status == nullptr || (which == 2 && flag == nullptr))
    return VT_ERR_INVALID_ARG;
  vt::selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      which, limit, reinterpret_cast<const unsigned*>(flag), dev_status);
  VT_RETURN_IF_LAUNCH_FAILED();
  return VT_OK;
}
