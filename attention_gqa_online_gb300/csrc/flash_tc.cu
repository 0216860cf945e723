// flash_tc.cu -- tcgen05 tensor-core flash kernel (TF32 / bf16 operands).
#include "common.cuh"
#include "internal.h"

namespace attn {

bool flash_tc_supported(const FlashArgs&, int) { return false; }

int launch_flash_tc(const FlashArgs&, int, cudaStream_t) { return ATTN_ERR_UNSUPPORTED; }

}  // namespace attn
