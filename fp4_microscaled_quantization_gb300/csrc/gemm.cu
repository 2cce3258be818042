// gemm.cu -- block-scaled 4-bit GEMM (placeholder until the tcgen05 kernel lands).
#include <stdint.h>
#include "../../include/fp4q.h"
extern "C" int32_t fp4q_gemm(const fp4q_operand*, const fp4q_operand*, int64_t, int64_t, int64_t, int32_t,
                             int32_t, void*, float*, uint32_t*, void*) {
  return FP4Q_ERR_UNSUPPORTED;
}
