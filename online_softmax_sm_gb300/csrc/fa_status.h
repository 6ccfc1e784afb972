// fa_status.h -- a device status value beside those of fa_internal.h, used
// by the backward kernels and decoded by fa_get_device_status.
#pragma once

namespace fa {

// A kernel's dynamic shared memory base was not aligned as its layout needs
// (the backward kernels fill the 227 KB limit and have no room to realign);
// the kernel wrote nothing.
constexpr int kDevLayout = 3;

}  // namespace fa
