// Precondition checks of debug builds (compiled with GDN_DEBUG_CHECKS).
//
// The operator contract lets one call update many requests' states in a
// shared pool ("[CUDA] Add compact GatedDeltaNet operator", Description:
// per-request state slots; "Replay compact fixed state for hybrid decoding",
// Key changes: replay from the committed bank into the inactive one).  Two
// requests of one call that write the same slot, or a replay that writes a
// slot another request of the call reads, race.  That is a caller error the
// release build does not look for (it would cost a launch per call); a debug
// build runs this kernel ahead of each call's work and reports it as
// GDN_DEVERR_DUP_SLOT in the status word (nothing is skipped).
#include "gdn_internal.cuh"

namespace gdn {

#ifdef GDN_DEBUG_CHECKS

namespace {

constexpr int DC_NT = 256;

// written[i] == written[j] for i != j, or written[i] == read[j] for i != j
// (read may be null), over n requests; slots outside [0, num_slots) are
// left to the kernels that own them.
__global__ void __launch_bounds__(DC_NT) distinct_slots_kernel(const int32_t *written, const int32_t *read, int n,
                                                               int num_slots, int32_t *status) {
    dependent_prologue();
    bool dup = false;
    for (int i = blockIdx.x * DC_NT + threadIdx.x; i < n; i += gridDim.x * DC_NT) {
        const int w = written[i];
        if (w < 0 || w >= num_slots) continue;
        for (int j = 0; j < n && !dup; ++j) {
            if (j == i) continue;
            dup = (j > i && written[j] == w) || (read && read[j] == w);
        }
    }
    if (dup) flag_error(status, GDN_DEVERR_DUP_SLOT);
}

}  // namespace

cudaError_t debug_check_distinct_slots(const int32_t *written, const int32_t *read, int n, int num_slots,
                                       int32_t *status, cudaStream_t stream) {
    if (!written || !status || n < 2) return cudaSuccess;
    const int blocks = (n + DC_NT - 1) / DC_NT;
    return launch_dependent(distinct_slots_kernel, dim3((unsigned)(blocks < 1024 ? blocks : 1024)), dim3(DC_NT), 0,
                            stream, written, read, n, num_slots, status);
}

#endif  // GDN_DEBUG_CHECKS

}  // namespace gdn
