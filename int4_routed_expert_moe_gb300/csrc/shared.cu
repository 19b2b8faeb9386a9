// Non-routed FP16 SwiGLU FFN ("Horizon RunMap -- Prévia Técnica",
// "03 / Arquitetura": the parts outside the routed experts stay FP16).
#include "common.h"
#include "kernels.h"

extern "C" size_t moe_shared_workspace_bytes(int T, int H, int Is) {
  if (T < 0 || H <= 0 || Is <= 0) return 0;
  return moe::kWorkspaceHeader + (size_t)T * Is * 2;
}

extern "C" int moe_shared_forward(const void* x, int T, int H, int Is, const void* wg,
                                  const void* wu, const void* wd, void* y, void* ws,
                                  size_t ws_bytes, void* stream) {
  moe::clear_error();
  (void)x; (void)T; (void)H; (void)Is; (void)wg; (void)wu; (void)wd; (void)y; (void)ws;
  (void)ws_bytes; (void)stream;
  return moe::fail(MOE_ERR_UNSUPPORTED, "moe_shared_forward: not built yet");
}
