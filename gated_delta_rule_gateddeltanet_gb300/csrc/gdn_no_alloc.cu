// gdn_forward_no_alloc: gdn_forward for callers that cannot allocate device
// memory.
//
// Some hosts own every byte of device memory through their own allocator and
// only hand an operator the inputs and outputs it declared -- an inference
// runtime's custom-operator interface, or a serving loop whose memory plan is
// fixed before it starts -- so there is nobody to ask for the chunked
// kernel's workspace; others run on latency-critical paths where a
// cudaMalloc, which may synchronise the device, is not acceptable.  This entry
// point takes the workspace from a fixed array compiled into the library
// instead of from the caller.  That array holds the chain list of the
// single-kernel chunked evaluation (the two-phase one needs per-chunk records
// that grow with the batch), so long sequences run on that kernel here.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (16 KiB) until the process exits.  In host code its name is
// only a host-side stand-in, not a device address, so the first call on each
// device looks the real address up (cudaGetSymbolAddress, with that device
// current) and caches it; make that first call before any stream capture.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// The cached address belongs to the device's primary context as it was at the
// first call: after cudaDeviceReset (or anything else that tears that context
// down) it is stale, so the library must not be used across a device reset.
//
// The sequence-parallel split plan has no single-kernel form (it needs
// per-sequence states and identity-run rows that grow with the batch), so it
// is refused here with GDN_ERR_UNSUPPORTED before anything else is looked at.
//
// All calls share the one array.  Everything the kernels need from it (the
// work counter and the chain list) is rewritten at the start of every call,
// so what an earlier call left there does not matter; but calls that overlap
// on the GPU (different streams, or different host threads without ordering)
// race on it and must not be issued.
#include <mutex>

#include "gdn_internal.cuh"

namespace {

static __device__ __align__(256) int32_t g_no_alloc_scratch[GDN_NO_ALLOC_MAX_SEQS + 2];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once per device).
gdn_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_no_alloc_scratch) != cudaSuccess || !ptr) return GDN_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_forward_no_alloc(const gdn_forward_args *args, gdn_stream_t stream) {
    if (!args) return GDN_ERR_NULL;
    if (args->plan == GDN_PLAN_CHUNKED_SPLIT) return GDN_ERR_UNSUPPORTED;
    size_t need = 0;
    gdn_status st = gdn::single_kernel_workspace_size(args, &need);
    if (st != GDN_OK) return st;
    if (need > sizeof(g_no_alloc_scratch)) return GDN_ERR_WORKSPACE;  // more than GDN_NO_ALLOC_MAX_SEQS sequences
    gdn_forward_args a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    if (need > 0) {
        void *ptr = nullptr;
        st = scratch_address(&ptr);
        if (st != GDN_OK) return st;
        a.workspace = ptr;
        a.workspace_bytes = sizeof(g_no_alloc_scratch);
    }
    return gdn_forward(&a, stream);
}
