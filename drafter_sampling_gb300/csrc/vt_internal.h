// Entry points shared between translation units of libvt (not exported).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace vt {

// vt_draft_step with two choices: status_reset = 1 zeroes *dev_status first
// (vt_draft_step), 0 adds this step's flags to it (later steps of a block);
// hidden_ready = 1 promises that no kernel still running in the stream writes
// the hidden states (they were complete before the previous kernel started),
// so the projection may stage them before its dependency wait.
int draft_step_impl(const uint16_t* hidden, int32_t B, int32_t H, const uint16_t* W_trim,
                    const int32_t* trim_ids, int32_t K, const float* uniforms, float temperature,
                    float* q, int64_t ldq, int32_t* tokens, int64_t ld_tokens,
                    int32_t* dev_status, void* workspace, size_t workspace_bytes, void* stream,
                    int status_reset, int hidden_ready);

}  // namespace vt
