// Host-side internals shared by the library's entry points (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

namespace gdn {

// The calling thread's record of the CUDA error behind its last GDN_ERR_LAUNCH or
// GDN_ERR_ALLOC (what gdn_last_cuda_error returns).  set_cuda_error records `e` and
// returns `code`; clear_cuda_error resets the record at the start of a call.
int set_cuda_error(cudaError_t e, int code);
void clear_cuda_error();

// Take the calling thread's pending gdn_set_phase_events hook (and clear it).
void take_phase_events(cudaEvent_t (&ev)[3]);

// Device address of the fixed scratch array behind gdn_prefill_static on device `dev`,
// or nullptr while no call on that device has looked it up.
void* static_scratch_address(int dev);

// Test hook behind gdn_debug_fail_allocations: true when the next library allocation
// is to fail (and counts it down).
bool take_injected_alloc_failure();

}  // namespace gdn
