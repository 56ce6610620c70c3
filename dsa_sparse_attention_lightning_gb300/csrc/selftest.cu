// selftest.cu -- dsa_selftest_bounded_wait: a library self-test that makes one
// bounded mbarrier wait run out on purpose.
//
// Every pipeline kernel of the library waits on mbarriers with a limit; when a
// limit runs out the kernel raises DSA_DEV_TIMEOUT in the status word, lets the
// copies it issued land, frees its tensor memory and returns, so that the
// context stays usable and the host learns of the failure through
// dsa_check_device_status.  That exit path never runs in a healthy pipeline.
// This kernel takes it deliberately: warp 0 holds a TMEM allocation, thread 0
// has a bulk copy in flight on one barrier and then waits on a second barrier
// that nothing ever arrives on, with a short limit chosen by the caller.  No
// fault, trap or assert is involved: the wait simply gives up.
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kSelftestCopyBytes = 256;
constexpr uint32_t kSelftestTmemCols = 32;

__global__ void __launch_bounds__(64, 1)
    selftest_wait_kernel(const uint8_t* src, uint8_t* echo, long long limit, uint32_t* status) {
  __shared__ __align__(128) uint8_t buf[kSelftestCopyBytes];
  __shared__ __align__(8) uint64_t copy_bar;   // completes when the bulk copy has landed
  __shared__ __align__(8) uint64_t never_bar;  // nothing ever arrives on it
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(&copy_bar, 1);
    mbar_init(&never_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, kSelftestTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  bool landed = false;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&copy_bar, kSelftestCopyBytes);
    bulk_g2s(buf, src, kSelftestCopyBytes, &copy_bar);
    mbar_wait(&never_bar, 0, status, limit);    // runs out: raises DSA_DEV_TIMEOUT
    // Drain before the CTA (and its shared memory) goes away.
    landed = mbar_wait(&copy_bar, 0, status, limit);
  }
  // The copied bytes go back out, so the host can see that the copy issued
  // before the failed wait completed and was read after it.
  if (__syncthreads_or(landed) && threadIdx.x < kSelftestCopyBytes / 4)
    reinterpret_cast<uint32_t*>(echo)[threadIdx.x] = reinterpret_cast<const uint32_t*>(buf)[threadIdx.x];
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_base, kSelftestTmemCols);
}

}  // namespace

// Layout of the self-test workspace: [0,256) status word, [256,512) copy
// source, [512,768) copy echo.
constexpr size_t kSelftestWorkspaceBytes = 768;

cudaError_t launch_selftest_wait(void* workspace, long long limit_cycles, cudaStream_t st) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  selftest_wait_kernel<<<1, 64, 0, st>>>(ws + 256, ws + 512, limit_cycles,
                                         reinterpret_cast<uint32_t*>(ws));
  return cudaGetLastError();
}

size_t selftest_workspace_bytes() { return kSelftestWorkspaceBytes; }

}  // namespace dsa
