// Driver-API entry points that libft calls through the CUDA runtime's
// entry-point lookup, so the library needs no link-time libcuda and still
// loads on a machine without a GPU driver (the ABI tests do that).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace ft {

// The function `name` of the installed driver (ABI of CUDA 12.0 or later),
// or nullptr if the lookup failed.  Looked up once per name and cached.
void* driver_fn(const char* name);

// The calling thread's current context, or nullptr.
CUcontext current_context();

}  // namespace ft
