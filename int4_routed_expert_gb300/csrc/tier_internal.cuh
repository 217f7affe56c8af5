// Internal entry points the expert tier (tier.cu) uses from the layer
// (capi.cu) and the SIMT batch kernels (gemv.cu).
#pragma once

#include "moe_internal.cuh"

namespace moe {

// moe_layer_create for a layer whose routed arrays hold `routed_experts`
// experts (the tier's HBM slots) instead of cfg->n_experts: the same checks,
// with the routed extents sized for the slots; the tensor-core maps are not
// made (the tier runs the SIMT batch kernels only).  Messages go to
// moe_last_error(NULL).
moe_status_t layer_create_slots(const moe_config_t* cfg, const moe_weights_t* w,
                                int routed_experts, moe_layer_t** out);

// The argument checks of moe_forward (and moe_route when y == nullptr and
// route_only is set), with x and y resolved to addresses the kernels use.
// Messages go to the layer's moe_last_error.
moe_status_t layer_check_call(moe_layer* h, const void** x, moe_dtype_t dt, int T, float** y,
                              const float* gamma, int accumulate, const moe_plan_t* plan,
                              bool route_only);

// Routing of moe_forward's batch paths into the workspace: prep, logits,
// selection, plan.
cudaError_t layer_route(moe_layer* h, const void* x, moe_dtype_t dt, int T, const float* gamma,
                        float eps, cudaStream_t s);

// Copies the workspace's plan to the caller's plan buffers (NULL: nothing).
cudaError_t layer_copy_plan(moe_layer* h, int T, const moe_plan_t* p, cudaStream_t s);

// SIMT batch kernels over the experts whose slot-table entry has the given
// phase: slot_tab[e] = (phase << kSlotPhaseShift) | slot.  The shared expert
// runs with phase 0.  Outputs land in the workspace rows of the plan, as for
// launch_gate_up / launch_down.
constexpr int kSlotPhaseShift = 24;
cudaError_t launch_gate_up_slots(const moe_weights_t& w, const Shape& sh, int T,
                                 const Workspace& ws, const int32_t* slot_tab, int phase,
                                 cudaStream_t s);
cudaError_t launch_down_slots(const moe_weights_t& w, const Shape& sh, int T, const Workspace& ws,
                              const int32_t* slot_tab, int phase, cudaStream_t s);

}  // namespace moe
