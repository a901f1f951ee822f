// Status names and version of the C ABI.
#include "common.h"

extern "C" {

const char* sgl_status_string(int status) {
    switch (status) {
        case SGL_OK: return "SGL_OK";
        case SGL_ERR_INVALID_ARG: return "SGL_ERR_INVALID_ARG";
        case SGL_ERR_NO_SLOTS: return "SGL_ERR_NO_SLOTS";
        case SGL_ERR_UNSUPPORTED: return "SGL_ERR_UNSUPPORTED";
        case SGL_ERR_CUDA: return "SGL_ERR_CUDA";
        case SGL_ERR_BOUNDS: return "SGL_ERR_BOUNDS";
        case SGL_ERR_STATE: return "SGL_ERR_STATE";
        case SGL_ERR_WORKSPACE: return "SGL_ERR_WORKSPACE";
        default: return "SGL_ERR_UNKNOWN";
    }
}

const char* sgl_version(void) { return "sglattn 0.1.0 (sm_103a)"; }

}  // extern "C"
