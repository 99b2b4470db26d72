// Self-test of the bounded device waits every kernel of this library uses.
//
// No kernel traps or spins without limit: a wait on an mbarrier phase that
// does not complete gives up after about a second (sm100_ptx.cuh), and the
// kernel then records DDT_ST_TIMEOUT for its sequence and leaves. This entry
// point runs that mechanism on its own, in one small kernel: a wait on a
// barrier that nothing arrives on (it must give up and report the timeout),
// then a wait on a phase that has completed (it must succeed at once). The
// GPU stays usable; the host reads the outcome.
#include "ddt_internal.cuh"
#include "sm100_ptx.cuh"

namespace ddt {
namespace {

using namespace sm100;

__global__ void k_wait_selftest(int32_t* out) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const unsigned long long t0 = global_ns();
  const bool first = mbar_wait(b, 0);  // nothing arrives: gives up
  const unsigned long long t1 = global_ns();
  mbar_arrive(b);                       // complete phase 0
  const bool second = mbar_wait(b, 0);  // completed: returns at once
  out[0] = first ? 0 : DDT_ST_TIMEOUT;
  out[1] = second ? 0 : DDT_ST_TIMEOUT;
  out[2] = (int32_t)((t1 - t0) / 1000000ull);  // milliseconds the first wait lasted
}

}  // namespace
}  // namespace ddt

extern "C" int ddt_wait_selftest(int32_t* result, cudaStream_t stream) {
  if (result == nullptr) return DDT_EINVAL;
  ddt::k_wait_selftest<<<1, 32, 0, stream>>>(result);
  return cudaGetLastError() == cudaSuccess ? DDT_OK : DDT_ELAUNCH;
}
