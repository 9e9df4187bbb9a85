// Dispatch -> per-expert SwiGLU FFN -> combine (xLLM MegaMoe pull request).
#include "internal.h"

extern "C" moe_status_t moe_dispatch_ffn_combine(const moe_config_t*, const void*, const int32_t*, const uint8_t*,
                                                 const float*, const void*, const void*, const void*, void*, void*,
                                                 size_t, void*) {
  return MOE_ERR_UNSUPPORTED;
}
