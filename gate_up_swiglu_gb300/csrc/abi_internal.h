// abi_internal.h -- shared between the library's translation units, not part
// of the public ABI.
#pragma once

namespace swiglu_abi {
// Remember a CUDA error for swiglu_last_cuda_error() (per calling thread).
__attribute__((visibility("hidden"))) void record_cuda_error(int err);
}  // namespace swiglu_abi
