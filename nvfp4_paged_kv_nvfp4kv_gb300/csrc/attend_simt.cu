// attend_simt.cu -- CUDA-core variant of the attention kernel (not built yet).
#include "internal.h"

namespace nvfp4kv {

bool attend_config_simt(int, int, int, AttendConfig*) { return false; }

}  // namespace nvfp4kv
