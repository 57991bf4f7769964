// qnn_internal.h -- host-side helpers shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "qnn.h"

namespace qnn {

// Device address of the status word that kernels set when a bounded wait
// gives up, for the current device (looked up once per device); nullptr if
// the lookup failed.
uint32_t *status_word();

// Number of SMs of the current device (cached per device).
int sm_count();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Maps the launch error (if any) of the last kernel launch to a status.
inline qnn_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? QNN_OK : QNN_ERR_CUDA;
}

// Code range of a quantized type.
inline bool qrange(int dt, int narrow, int32_t *lo, int32_t *hi)
{
    switch (dt) {
    case QNN_S8: *lo = narrow ? -127 : -128; *hi = 127; return true;
    case QNN_U8: *lo = 0; *hi = 255; return true;
    case QNN_S4: *lo = narrow ? -7 : -8; *hi = 7; return true;
    case QNN_U4: *lo = 0; *hi = 15; return true;
    default: return false;
    }
}

}  // namespace qnn
