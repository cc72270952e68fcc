// Host-side helpers shared by the libpkv entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Status of the launches just issued on this thread.
inline int launch_status() { return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace pkv
