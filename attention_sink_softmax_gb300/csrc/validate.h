// validate.h - argument checks shared by every C entry point of libsinkattn
// (api.cu and the no-allocation entry point in noalloc.cu).
#pragma once

#include "../../include/sink_attn.h"

namespace sinkattn {

// Field checks of sink_attn_params_t, identical for every entry point that
// takes one: SINK_ERR_INVALID_ARG for inconsistent or out-of-range fields,
// SINK_ERR_UNSUPPORTED for valid shapes no kernel here takes.
sink_status_t validate_params(const sink_attn_params_t* p);

}  // namespace sinkattn
