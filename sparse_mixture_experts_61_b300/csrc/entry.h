// Internal forms of the forward entry points (moe_api.cu), shared with the
// host-batch pipeline (host_pipeline.cu).  Each runs the exported call's full
// host-side validation; the mode then decides what is enqueued.
#pragma once

#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

enum class EntryMode {
  kValidate,   // validation only, nothing enqueued
  kRun,        // clear the device flag word, then enqueue the layer (the exported call)
  kRunKeepFlags  // enqueue the layer; flags raised by earlier calls on this workspace stay
};

moe_status forward_entry(const moe_config* cfg, const moe_forward_args* a, void* ws,
                         size_t ws_bytes, cudaStream_t st, EntryMode mode);

moe_status ec_forward_entry(const moe_config* cfg, const moe_expert_choice_args* a, void* ws,
                            size_t ws_bytes, cudaStream_t st, EntryMode mode);

}  // namespace moe
