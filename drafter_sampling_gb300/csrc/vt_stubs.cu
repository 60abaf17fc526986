#include "vt_common.cuh"
extern "C" size_t vt_calibrate_topk_workspace_bytes(int64_t, int32_t, int32_t) { return 256; }
extern "C" int vt_calibrate_topk(const int32_t*, int64_t, int32_t, int32_t, uint32_t*, int32_t*, int32_t*, void*, size_t, void*) { return VT_ERR_UNSUPPORTED; }
extern "C" int vt_trim_head(const uint16_t*, int32_t, int32_t, const int32_t*, int32_t, uint16_t*, int32_t*, int32_t*, int32_t*, void*) { return VT_ERR_UNSUPPORTED; }
extern "C" size_t vt_draft_workspace_bytes(int32_t, int32_t, int32_t) { return 256; }
extern "C" int vt_draft_logits(const uint16_t*, int32_t, int32_t, const uint16_t*, int32_t, float, float*, int64_t, void*, size_t, void*) { return VT_ERR_UNSUPPORTED; }
extern "C" int vt_draft_step(const uint16_t*, int32_t, int32_t, const uint16_t*, const int32_t*, int32_t, const float*, float, float*, int64_t, int32_t*, int32_t*, void*, size_t, void*) { return VT_ERR_UNSUPPORTED; }
