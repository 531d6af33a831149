// Library identity and status texts.
#include "pa.h"

extern "C" {

const char* pa_version(void) { return "paged_kv_cache_124_gb300 0.1 (sm_103a)"; }

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_FAIL_NO_BLOCKS: return "no free blocks (nothing changed)";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape";
        case PA_ERR_MISALIGNED: return "pointer not aligned";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_UNKNOWN_SEQ: return "unknown sequence";
        case PA_ERR_DUPLICATE_SEQ: return "sequence already exists";
        case PA_ERR_SWAPPED: return "sequence is swapped out";
        default: return "unknown status";
    }
}

}  // extern "C"
