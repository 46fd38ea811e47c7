// Internal forms of the forward entry points (moe_api.cu), shared with the
// host-batch pipeline (host_pipeline.cu).  Each runs the exported call's full
// host-side validation; the mode then decides what is enqueued.
#pragma once

#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {

// The first bytes of a forward workspace (moe_workspace_size, moe_stage_workspace_size,
// moe_expert_choice_workspace_size): the device flag word, then the split-tile counters
// of the layer's two expert GEMMs.  Every exported call that starts a layer's work
// zeroes this whole region first.
constexpr size_t kFlagRegionBytes = 256 + 2 * kSplitCounters * sizeof(int);
static_assert(kFlagRegionBytes % 256 == 0, "regions after it stay 256-byte aligned");
static_assert(kFlagRegionBytes == 5376, "include/moe.h states this size");

enum class EntryMode {
  kValidate,   // validation only, nothing enqueued
  kRun,        // clear the flag region, then enqueue the layer (the exported call)
  kRunKeepFlags  // enqueue the layer; flags raised by earlier calls on this workspace stay
                 // (the caller cleared the flag region before the first of them)
};

// Validation of a moe_config shared by every forward-side entry point: types and
// modes in range (MOE_ERR_INVALID_ARGUMENT), sizes in the supported range
// (MOE_ERR_UNSUPPORTED).
moe_status check_config(const moe_config* c);

moe_status forward_entry(const moe_config* cfg, const moe_forward_args* a, void* ws,
                         size_t ws_bytes, cudaStream_t st, EntryMode mode);

moe_status ec_forward_entry(const moe_config* cfg, const moe_expert_choice_args* a, void* ws,
                            size_t ws_bytes, cudaStream_t st, EntryMode mode);

}  // namespace moe
