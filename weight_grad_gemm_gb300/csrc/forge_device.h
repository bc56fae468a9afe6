// forge_device.h -- the device check every entry point makes (defined in
// forge_api.cu).
#pragma once
#include "forge.h"

namespace forge {

// The current device, checked once per device for compute capability 10.3;
// on success *sms receives its SM count.
forge_status device_sms(int* sms);

}  // namespace forge
