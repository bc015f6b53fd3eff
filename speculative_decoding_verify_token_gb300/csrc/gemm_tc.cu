// tcgen05 GEMM (bf16 models): placeholder until the tensor-core path lands.
#include "model.h"
#include "host_util.h"

namespace sv {
int tc_create(Ctx& c) { c.use_tc = false; return SPEC_OK; }
void tc_destroy(Ctx& c) { (void)c; }
int tc_gemm(Ctx& c, int, int, const void*, int, const EpiArgs&, cudaStream_t) {
    (void)c;
    return set_error(SPEC_E_STATE, "tensor-core GEMM not available");
}
}  // namespace sv
