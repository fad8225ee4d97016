// ce_host.cuh -- host-side helpers shared by the C-ABI units: ce_api.cu (the
// cross-entropy rows, where they are defined) and ce_api_tc.cu (the
// tensor-core entry points).
#pragma once

#include <cstdint>

#include "../../include/ce_gb300.h"

namespace ce_host {

// The current device's SM count and the address of its error word (bit 0: a
// target outside [0, V); bit 1: a bounded wait ran out).
struct DeviceInfo {
  int sm_count = 0;
  unsigned int* err = nullptr;
};

// DeviceInfo of the current device (looked up once per device); its index in *dev_out.
ce_status device_info(DeviceInfo& out, int* dev_out);

// Suspend-time hint of the kernels' mbarrier waits (ns).
unsigned int wait_hint_ns();

// Adds n to the library's launch counter (ce_launch_count).
void count_launches(uint64_t n);

}  // namespace ce_host
