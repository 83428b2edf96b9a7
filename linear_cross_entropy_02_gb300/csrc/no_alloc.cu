// flce_ce_only_noalloc: the CE-only pass with its scratch memory in a
// file-scope device array instead of a caller-provided workspace.
//
// Who needs this: callers that cannot call cudaMalloc (or any allocating
// routine) at the point where they need the loss - for example code running
// inside a custom allocator's own callbacks, a framework hook that runs while
// the allocator is locked, or an embedding that forbids device allocations
// after start-up because it has budgeted every byte. They still own their
// inputs and outputs; only the scratch comes from here.
//
// Costs and rules:
//  - Every GPU on which this module is loaded keeps kStaticScratchBytes
//    (64 MiB) reserved until the process exits.
//  - The first call on each device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current). Make that first call
//    before any stream capture.
//  - All calls on a device share the one array and it keeps the previous
//    call's contents. The prologue kernel re-initialises every field that must
//    start at zero (status word, counters, sums), and every other byte is
//    written before it is read. Calls whose work overlaps on the GPU (other
//    streams, other host threads) race on the array: serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "flce.h"
#include "flce_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_flce_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

__global__ void copy_status_kernel(const flce::Header* hdr, int32_t* out) { *out = hdr->status; }

// Device address of the array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_flce_static_scratch) != cudaSuccess || p == nullptr) return FLCE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" int flce_ce_only_noalloc(const flce_params* p, const void* h, const void* W, const int64_t* labels,
                                    float* loss, float* token_accuracy, int32_t* device_status, void* stream) {
  if (p == nullptr) return FLCE_ERR_ARG;
  flce_params q = *p;
  size_t need = 0;
  if (q.chunk_rows == 0) {
    // Largest chunk (8192, 4096, ..., 128 rows) whose scratch fits the array.
    for (int64_t c = 8192; c >= 128; c /= 2) {
      q.chunk_rows = c;
      need = flce_workspace_size(&q, FLCE_MODE_CE_ONLY, 0, 0);
      if (need == 0 || need <= kStaticScratchBytes) break;
    }
  } else {
    need = flce_workspace_size(&q, FLCE_MODE_CE_ONLY, 0, 0);
  }
  if (need == 0) return FLCE_ERR_ARG;
  if (need > kStaticScratchBytes) return FLCE_ERR_WORKSPACE;  // vocabulary too large for the fixed array
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != FLCE_OK) return rc;
  rc = flce_ce_only(&q, h, W, labels, loss, token_accuracy, scratch, kStaticScratchBytes, stream);
  if (rc != FLCE_OK) return rc;
  if (device_status != nullptr) {
    copy_status_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const flce::Header*>(scratch), device_status);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}
