// Temporary: the streamed stack is filled in by the stack scheduler.
#include "common.cuh"
using namespace sl;
struct sl_stack { int dummy; };
extern "C" {
sl_status sl_stack_blob_layout(int32_t, int64_t, int64_t, int64_t, size_t*, size_t*) { return set_error(SL_ERR_UNSUPPORTED, "not built yet"); }
sl_status sl_stack_create(const sl_stack_desc*, sl_stack**, size_t*, size_t*) { return set_error(SL_ERR_UNSUPPORTED, "not built yet"); }
sl_status sl_stack_destroy(sl_stack*) { return SL_OK; }
size_t sl_stack_workspace_size(const sl_stack*, int64_t, int32_t) { return 0; }
sl_status sl_stream_stack_step(sl_stack*, int32_t, const float*, int64_t, const float*, const void* const*, const void* const*, int32_t, float, float*, float*, float* const*, float* const*, void*, size_t, cudaStream_t) { return set_error(SL_ERR_UNSUPPORTED, "not built yet"); }
sl_status sl_stack_last_step_stats(const sl_stack*, uint64_t*, uint64_t*) { return set_error(SL_ERR_UNSUPPORTED, "not built yet"); }
}
