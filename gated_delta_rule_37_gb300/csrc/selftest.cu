// Diagnostic: exercise the library's bounded-wait path on purpose.  One CTA
// waits on an mbarrier that nothing ever arrives on, with the same bounded wait
// (tc::mbar_wait: %globaltimer limit) the tensor-core kernels use; when the
// wait gives up, the kernel records the failure in the device error word and
// returns, so the host reads GDR_ERR_DEVICE_TIMEOUT from gdr_get_device_status
// and the context stays usable.  No fault, trap or unbounded loop is involved.
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

#include "gdr.h"

namespace gdr {
namespace {

constexpr unsigned kSelftestCode = 0x100u;  // error-word bit of this diagnostic

__global__ void bounded_wait_selftest_kernel(unsigned int* err) {
    __shared__ uint64_t mbar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(tc::smem_u32(&mbar), 1);  // one arrival would complete it; none comes
        abort_flag = 0;
        tc::mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(tc::smem_u32(&mbar), 0, &abort_flag)) atomicOr(err, kSelftestCode);
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" int gdr_selftest_bounded_wait(gdr_stream_t stream) {
    unsigned int* err = device_error_word();
    if (!err) return set_last_error(GDR_ERR_LAUNCH, "error word unavailable");
    bounded_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_last_error(GDR_ERR_LAUNCH, "selftest launch: %s", cudaGetErrorString(e));
    return set_last_error(GDR_OK, "");
}
