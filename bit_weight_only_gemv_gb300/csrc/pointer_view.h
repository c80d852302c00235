// Host helper shared by the slot pools (slot_pool.cu, dev_pool.cu).
#pragma once

namespace w4 {

// The address through which kernels on the current device read `ptr`: the
// pointer itself for memory of this device (or managed memory), the mapped
// address of page-locked host memory, nullptr for anything else (pageable
// host memory, another device's memory), which only the copy engine serves.
const void* device_view(const void* ptr);

}  // namespace w4
