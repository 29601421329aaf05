// Internal interface of the attention core (attn.cu) for the block scheduler.
// Not part of the public ABI; the C entry points are in include/boostattn.h.
#pragma once

#include "../../include/boostattn.h"
#include "gemm.h"

namespace bn {

// BN_OK, or the status bn_attn_forward would return for these shapes
bn_status attn_check(const bn_attn_desc& d);
// fp32 values of the backward's row terms (D and lse log2(e)): 2 B H Lp
size_t attn_scratch_floats(const bn_attn_desc& d);
// One launch on c.stream: o and lse ([B H, Lp] fp32) from q, k, v.
cudaError_t attn_forward(Ctx& c, const bn_attn_desc& d, const void* q, const void* k,
                         const void* v, void* o, float* lse, int* status);
// Three launches: the row terms into rows_scratch (attn_scratch_floats values),
// then dk and dv, then dq.
cudaError_t attn_backward(Ctx& c, const bn_attn_desc& d, const void* q, const void* k,
                          const void* v, const void* o, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv, float* rows_scratch, int* status);

}  // namespace bn
