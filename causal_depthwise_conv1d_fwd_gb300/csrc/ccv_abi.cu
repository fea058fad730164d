// Status strings and version of the ccv C ABI.
#include "ccv_common.cuh"

extern "C" const char *ccv_status_string(int status) {
    switch (status) {
        case CCV_OK: return "ok";
        case CCV_ERR_NULL_POINTER: return "a required pointer is NULL";
        case CCV_ERR_WIDTH: return "width must be in 2..5";
        case CCV_ERR_SIZE: return "a size is negative, inconsistent or too large";
        case CCV_ERR_STATE_LEN: return "conv_state has fewer columns than the method needs";
        case CCV_ERR_ALIAS: return "an output overlaps an input it may not alias";
        case CCV_ERR_STRIDE: return "a stride is negative";
        case CCV_ERR_RANGE:
            return "a stream's D-range [off_s, off_s+ws) leaves the cache or overlaps another stream's";
        case CCV_ERR_CAPACITY: return "an output buffer has fewer entries than the call needs";
        case CCV_ERR_ARGUMENT: return "has_initial_state needs conv_states";
        default: break;
    }
    if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown ccv status";
}

// 1.1.0: ccv_update_spec and paged_sconv_fwd_streams added.
// 1.2.0: programmatic dependent launches; short-problem prefill kernels.
// 1.3.0: paged_sconv_fwd_with_metadata added.
extern "C" int ccv_version(void) { return 1 * 10000 + 3 * 100 + 0; }
