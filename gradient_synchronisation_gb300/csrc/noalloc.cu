// zr_partition_static: the push-side h0 partition for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs inside a training framework's gradient
// communication hook, where the framework's caching allocator owns the device
// memory (a direct cudaMalloc there bypasses its accounting and its
// fragmentation control, and cudaMalloc / cudaFree can synchronise the
// device in the middle of the overlapped backward pass), and services that
// reserve every byte of device memory at start-up and forbid new allocations
// afterwards.  Such callers can own their inputs and outputs but not a
// per-call workspace, so this entry point takes its scratch from a fixed
// array compiled into the library instead.
//
// The scratch is a file-scope __device__ array of ZR_STATIC_SCRATCH_BYTES
// (every GPU that loads the library holds it until the process exits).  It
// holds the partition's per-(partition, CTA) count table and the status and
// grid-wait words, whose size does not depend on the list length, so every
// valid request fits.  Host code must not hand the array's name to a
// kernel: on the host that name is only a stand-in symbol.  Its device
// address is looked up once per device, on the first call made with that
// device current, with cudaGetSymbolAddress; that first call should
// therefore come before any stream capture.  The address is kept for the
// life of the process, so the entry point must not be used on a device after
// cudaDeviceReset (which reloads the module and can move the array).  Every
// call on a device shares the one array and clears the parts that must start
// at zero itself, so calls whose work overlaps on the GPU (different streams
// without ordering between them) race on it.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "zr.h"
#include "zr_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_partition_scratch[ZR_STATIC_SCRATCH_BYTES];

// Device address of g_partition_scratch, per device: null until the first
// call on that device looks it up (under the lock); read without the lock
// once set.
std::atomic<void*> g_scratch_address[64];
std::mutex g_scratch_lock;

zr_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ZR_ERR_CUDA;
  void* p = g_scratch_address[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> guard(g_scratch_lock);
    p = g_scratch_address[dev].load(std::memory_order_relaxed);
    if (!p) {
      if (cudaGetSymbolAddress(&p, g_partition_scratch) != cudaSuccess || !p) return ZR_ERR_CUDA;
      g_scratch_address[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return ZR_OK;
}

}  // namespace

extern "C" zr_status zr_partition_static(const int32_t* idx, const float* val, int64_t nnz,
                                         int32_t n_parts, uint64_t part_seed, int32_t* out_idx,
                                         float* out_val, int64_t* d_offsets, void* stream) {
  if (nnz < 0 || nnz > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS || !d_offsets)
    return ZR_ERR_INVALID_ARG;
  if (nnz > 0 && (!idx || !val || !out_idx || !out_val)) return ZR_ERR_INVALID_ARG;
  if (zr::partition_workspace_bytes(nnz, n_parts) > (size_t)ZR_STATIC_SCRATCH_BYTES)
    return ZR_ERR_CAPACITY;
  void* scratch = nullptr;
  const zr_status st = scratch_for_current_device(&scratch);
  if (st != ZR_OK) return st;
  return zr::partition_launch(idx, val, nnz, n_parts, part_seed, out_idx, out_val, d_offsets,
                              scratch, static_cast<cudaStream_t>(stream));
}
