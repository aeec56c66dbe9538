// bmm_rs_a2a_noalloc: the packed variant of the fused op with scratch memory
// that the library owns, for callers that cannot allocate device memory.
//
// The packed variant repacks operands whose rows lack a 16-byte pitch into
// scratch memory, then runs the TMA kernel on the copies.  bmm_rs_a2a_ex
// takes that scratch from the caller (the workspace option).  Some callers
// have no device allocator to take it from: a plugin inside a host program
// that owns all device memory and gives its plugins only their inputs and
// outputs, or code that must not call cudaMalloc because cudaMalloc may
// synchronise the device.  This entry point serves them from one
// file-scope device array of BRA_NOALLOC_SCRATCH_BYTES, loaded with the
// library's module on every device that uses it and held until the process
// exits.
#include <mutex>

#include "bra_internal.h"

namespace {

// The scratch array.  In host code this name is the host-side shadow of the
// device variable, not a device address; only the address obtained from
// cudaGetSymbolAddress (below) may be given to a kernel.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BRA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];   // device address of the array, per device

// The array's device address on the current device, looked up once per
// device (the first call on a device does it, with that device current).
int scratch_address(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BRA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BRA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress((void**)&p, g_noalloc_scratch) != cudaSuccess || !p)
      return BRA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *ptr = g_scratch_addr[dev];
  return BRA_OK;
}

}  // namespace

extern "C" int bmm_rs_a2a_noalloc(const void* const x[], const void* const weight[],
                                  const void* const bias[], int64_t ep, int64_t tp, int64_t E,
                                  int64_t C, int64_t M, int64_t H, int64_t yShardType,
                                  int dtype, void* const out[], int transpose_weight,
                                  bra_stream_t stream) {
  bra_fused_options o = {};
  o.transpose_weight = transpose_weight ? 1 : 0;
  o.variant = BRA_VARIANT_PACKED;
  // The same argument checks as bmm_rs_a2a_ex, then the scratch the copies
  // need (0 when the operands are TMA-ready and nothing is copied).
  const int64_t need = bmm_rs_a2a_workspace_size(x, weight, bias, ep, tp, E, C, M, H,
                                                 yShardType, dtype, out, &o);
  if (need < 0) return (int)-need;
  if (need > (int64_t)BRA_NOALLOC_SCRATCH_BYTES) return BRA_ERR_UNSUPPORTED;
  if (need > 0) {
    void* p = nullptr;
    const int rc = scratch_address(&p);
    if (rc != BRA_OK) return rc;
    o.workspace = p;
    o.workspace_bytes = (int64_t)BRA_NOALLOC_SCRATCH_BYTES;
  }
  // Nothing in the scratch has to start at zero: the repack writes every
  // byte the TMA maps read (columns past a row's length are read as zeros
  // by the maps' bounds, not from memory), so a previous call's contents
  // are harmless.
  return bmm_rs_a2a_ex(x, weight, bias, ep, tp, E, C, M, H, yShardType, dtype, out, &o, stream);
}
