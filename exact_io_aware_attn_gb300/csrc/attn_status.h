// attn_status.h -- the device status word shared by all kernels of libattn.
//
// Every kernel receives a pointer to one 32-bit word in device memory. A
// bounded wait that gives up stores (first error wins, atomicCAS from 0):
//   bits 0-7   status code (ATTN_ERR_TIMEOUT)
//   bits 8-15  kernel id
//   bits 16-23 wait site inside that kernel
// The host reads and clears the word through attn_get_device_error.
#pragma once

#include <cstdint>

namespace attn {

// Time limit of one device-side wait. Long enough that no healthy wait on
// a loaded GPU reaches it, short enough that a lost arrival ends the kernel
// within seconds instead of hanging the device.
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;

constexpr uint32_t kStatusTimeout = 4u;  // == ATTN_ERR_TIMEOUT

enum KernelId : uint32_t {
  kKernPrefill = 1, kKernDecodeSplit = 2, kKernDecodeCombine = 3, kKernSelftest = 4,
  kKernBwdKV = 5, kKernBwdQ = 6, kKernDecodePaged = 7
};

// A word for a status code other than a timeout (e.g. ATTN_ERR_INVALID_ARG
// for a block-table entry outside the page pool, found on the device).
__host__ __device__ constexpr uint32_t status_word_code(uint32_t code, uint32_t kernel,
                                                        uint32_t site) {
  return code | (kernel << 8) | (site << 16);
}

__host__ __device__ constexpr uint32_t status_word(uint32_t kernel, uint32_t site) {
  return kStatusTimeout | (kernel << 8) | (site << 16);
}

}  // namespace attn
