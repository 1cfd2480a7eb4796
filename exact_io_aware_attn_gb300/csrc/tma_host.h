// tma_host.h -- host helpers shared by the tensor-core kernels: TMA tensor
// maps over [BH][T][D] 16-bit tensors and the SM count of a device.
#pragma once

#include <cuda.h>

namespace attn {

// [BH][T][D] 16-bit tensor viewed as 3-D (D innermost), box 64 x box_rows x 1,
// 128-byte swizzle; rows past T read as zero. False if the driver entry point
// is missing or the encoding is rejected (base not 16-byte aligned, ...).
bool make_map(CUtensorMap* map, const void* base, int T, int BH, int D, bool bf16, int box_rows);

// Multiprocessor count of device `dev` (cached per device).
int device_sms(int dev);

}  // namespace attn
