// moe_align_noalloc: moe_align with its scratch in a fixed device array.
//
// moe_align needs a per-chunk histogram table once M*top_k exceeds 4096
// pairs, and its caller provides that table.  Some callers cannot: a plugin
// that a host runtime hands only its input and output tensors has no
// allocator of its own, and a caller on a latency-critical path cannot afford
// cudaMalloc/cudaFree, which may block or synchronise the device.  This entry
// point takes the table from a file-scope device array instead, so it
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
//
// Limit: the table is kNoAllocScratchBytes (1 MiB), i.e. ceil(M*top_k / 1024)
// chunks * E experts * 4 bytes must fit (for E = 384 that is up to 698,368
// routing pairs; for E = 1024, 262,144).  Larger calls are rejected before
// anything is launched.  Every GPU that loads the library holds the array
// until the process exits.
#include <mutex>

#include "moe_int4.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

// In host code this name stands for the device symbol; its device address is
// obtained with cudaGetSymbolAddress, per device, below.
static __device__ __align__(256) int32_t g_align_chunk_tab[kNoAllocScratchBytes / 4];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_align_chunk_tab on the current device, looked up once per
// device (the first call on each device that needs the table does this
// set-up).  The cached address belongs to the device's primary context: after
// cudaDeviceReset it is stale, so a process that resets a device does not call
// moe_align_noalloc with a table-sized routing on it again.
int noalloc_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_align_chunk_tab) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_align_noalloc(const int32_t *topk_ids, int M, int top_k, int E, int block_m,
                      int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
                      uint32_t *err_flags, moe_stream_t stream) {
    if (M < 0 || top_k < 1 || top_k > 32 || E < 1 || E > 1024 || block_m < 1 || block_m > 256)
        return MOE_ERR_SHAPE;
    if ((long long)M * top_k > (1LL << 30)) return MOE_ERR_SHAPE;
    const size_t need = moe_align_scratch_bytes(M, top_k, E);
    if (need > kNoAllocScratchBytes) return MOE_ERR_NOALLOC_LIMIT;
    if (need == 0)  // single-block align: no table, no device set-up
        return moe_align(topk_ids, M, top_k, E, block_m, sorted_ids, expert_ids, num_post_pad,
                         err_flags, nullptr, 0, stream);
    void *scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != MOE_OK) return rc;
    // The histogram pass writes every table entry that the later passes read,
    // so nothing left in the array by an earlier call needs clearing.
    return moe_align(topk_ids, M, top_k, E, block_m, sorted_ids, expert_ids, num_post_pad,
                     err_flags, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
