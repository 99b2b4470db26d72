// Verify attention (bf16 path) for callers that cannot allocate device memory.
//
// The regular entry point, ddt_verify_attn, takes its split-KV scratch from
// the caller (sized by ddt_verify_attn_workspace_size). Some callers have no
// way to provide it: code that runs where device allocation is not allowed
// or not available (for example a host program whose memory is entirely
// pre-reserved by another runtime, a plugin that receives only input and
// output buffers from its host application, or a latency-critical loop that
// must never enter the allocator). ddt_verify_attn_noalloc serves them by
// running the same kernels with the scratch taken from a fixed array that
// this library places in device memory when it is loaded.
//
// Costs and rules:
//  - the array (kScratchBytes) is reserved on every GPU that loads the
//    library and held until the process exits;
//  - a call whose split-KV scratch would exceed it is refused with
//    DDT_EWORKSPACE before anything is enqueued;
//  - every call uses the same array, so calls whose GPU work overlaps (other
//    streams, other host threads) race on it; serialise them;
//  - the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and keeps it for the
//    life of the process; make that first call before any stream capture.
//    Host threads may make first calls at the same time (the address is kept
//    in an atomic; racing lookups store the same value). A cudaDeviceReset
//    destroys the array with the context, and the kept address then points at
//    nothing: this entry point must not be used after a reset of its device;
//  - nothing in the array needs to start at zero: every partial result the
//    merge kernel reads is written earlier in the same call.
#include <atomic>

#include "ddt_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

// Device address of g_verify_scratch, looked up once per device.
constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

void* scratch_address(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  void* p = g_scratch_addr[device].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_addr[device].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace

extern "C" int ddt_verify_attn_noalloc(const ddt_attn_dims* dims, const void* q_lat,
                                       const void* q_pe, const void* kv_cache,
                                       const int32_t* block_table, const int32_t* prefix_len,
                                       const uint64_t* vis_bits, void* out, float* lse,
                                       int32_t* status, cudaStream_t stream) {
  int rc = ddt::check_verify_attn_args(dims, q_lat, q_pe, kv_cache, block_table, prefix_len,
                                       vis_bits, out, status);
  if (rc) return rc;
  if (dims->dtype != DDT_BF16) return DDT_EUNSUPPORTED;
  if (dims->kv_rows < 1) return DDT_EINVAL;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q_lat) | reinterpret_cast<uintptr_t>(q_pe) |
                        reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(out);
  if (mis & 15u) return DDT_EUNSUPPORTED;
  const size_t need = ddt::verify_attn_bf16_workspace(*dims);
  if (need > kScratchBytes) return DDT_EWORKSPACE;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return DDT_ELAUNCH;
  void* scratch = scratch_address(device);
  if (scratch == nullptr) return DDT_ELAUNCH;
  const cudaError_t e = ddt::launch_verify_attn_bf16(*dims, q_lat, q_pe, kv_cache, block_table,
                                                     prefix_len, vis_bits, out, lse, status,
                                                     scratch, kScratchBytes, stream);
  return e == cudaSuccess ? DDT_OK : DDT_ELAUNCH;
}
