// noalloc.cu -- moe_layer_forward_static: the whole layer with its scratch in a
// fixed device array owned by this library, for callers that cannot allocate
// device memory themselves.
//
// Who needs it: code that runs where cudaMalloc is off limits or unavailable --
// a custom allocator that hands out only the model's tensors, a serving loop
// that forbids allocation after start-up, an embedding host without access to
// a caching allocator -- and so cannot provide the workspace the other entry
// points take.  Those callers still pass inputs and outputs; only the scratch
// moves into the library.
//
// The array below is a static __device__ object: every GPU that loads this
// library holds its MOE_STATIC_SCRATCH_BYTES from module load until the
// process exits.  In host code its name is only a host-side stand-in for the
// symbol, not a device address, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current, and that
// address is what the launches get.
#include <mutex>

#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device (set-up on the
// first call per device).
moe_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_layer_forward_static(const moe_dims_t* dims, const void* x,
                                                 const void* router_w,
                                                 const moe_expert_weights_t* experts,
                                                 const moe_shared_weights_t* shared, void* out,
                                                 int32_t* topk_ids_out, float* topk_weights_out,
                                                 int32_t* device_status_out, void* stream) {
  // Every host-side check comes before anything is enqueued.
  moe_status_t s = moe::layer_precheck(dims, x, router_w, experts, shared, out, topk_ids_out,
                                       topk_weights_out);
  if (s != MOE_OK) return s;
  size_t need = 0;
  if ((s = moe_workspace_bytes(dims, &need)) != MOE_OK) return s;
  if (need > (size_t)MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  if (device_status_out && (reinterpret_cast<uintptr_t>(device_status_out) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  if (dims->T == 0) return MOE_OK;  // nothing enqueued, device_status_out untouched
  void* ws = nullptr;
  if ((s = scratch_address(&ws)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word is the only scratch that must start at zero.
  if ((s = moe_workspace_init(ws, (size_t)MOE_STATIC_SCRATCH_BYTES, stream)) != MOE_OK) return s;
  s = moe_layer_forward(dims, x, router_w, experts, shared, out, topk_ids_out, topk_weights_out,
                        ws, (size_t)MOE_STATIC_SCRATCH_BYTES, stream);
  if (s != MOE_OK) return s;
  if (device_status_out &&
      cudaMemcpyAsync(device_status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
