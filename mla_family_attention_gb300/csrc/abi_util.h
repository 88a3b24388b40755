// Host helpers of the C-ABI layer (defined in api.cu) that other entry-point
// files reuse: error reporting, device facts, test knobs, argument checks.
#pragma once

#include "../../include/mla.h"
#include "kernels.h"

namespace mla {

mla_status set_error(mla_status s, const char* msg);
mla_status current_device(DeviceInfo* out);
Knobs current_knobs();
mla_status check_decode_args(const void* q, const void* k, const void* v, const void* cu,
                             const void* gate, const void* out, int B, int H, int max_len,
                             float scale);

}  // namespace mla
