// Host-only parts of the ABI: diagnostics, the expert block layout and the
// pack/unpack copies between the canonical arrays and one block.
#include <cstring>
#include <string>

#include "common.h"

namespace moe {

static thread_local char g_last_error[512] = {0};

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

void clear_error() { g_last_error[0] = 0; }

const char* last_error() { return g_last_error; }

}  // namespace moe

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_ARG: return "MOE_ERR_ARG";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE";
    case MOE_ERR_STATE: return "MOE_ERR_STATE";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_INJECTED: return "MOE_ERR_INJECTED";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    default: return "MOE_ERR_UNKNOWN";
  }
}

const char* moe_last_error(void) { return moe::last_error(); }

int moe_version(void) { return 1; }

size_t moe_expert_block_bytes(const moe_expert_shape* s) {
  if (!moe::valid_shape(s)) return 0;
  return moe::block_layout(s->hidden, s->inter, s->group).total;
}

int moe_expert_block_offsets(const moe_expert_shape* s, size_t off[9]) {
  moe::clear_error();
  if (!off) return moe::fail(MOE_ERR_ARG, "offsets_out is NULL");
  if (!moe::valid_shape(s)) return moe::fail(MOE_ERR_SHAPE, "invalid expert shape");
  const moe::BlockLayout b = moe::block_layout(s->hidden, s->inter, s->group);
  const size_t v[9] = {b.q_gate, b.q_up, b.q_down, b.s_gate, b.z_gate,
                       b.s_up, b.z_up, b.s_down, b.z_down};
  for (int i = 0; i < 9; ++i) off[i] = v[i];
  return MOE_OK;
}

int moe_pack_expert(const moe_expert_shape* s, const uint8_t* q_gate,
                    const uint8_t* q_up, const uint8_t* q_down,
                    const uint16_t* s_gate, const uint16_t* z_gate,
                    const uint16_t* s_up, const uint16_t* z_up,
                    const uint16_t* s_down, const uint16_t* z_down,
                    void* block_out) {
  moe::clear_error();
  if (!moe::valid_shape(s)) return moe::fail(MOE_ERR_SHAPE, "invalid expert shape");
  if (!q_gate || !q_up || !q_down || !s_gate || !z_gate || !s_up || !z_up ||
      !s_down || !z_down || !block_out)
    return moe::fail(MOE_ERR_ARG, "NULL array");
  const moe::BlockLayout b = moe::block_layout(s->hidden, s->inter, s->group);
  uint8_t* o = static_cast<uint8_t*>(block_out);
  const size_t qgu = b.q_up - b.q_gate, qd = b.s_gate - b.q_down;
  const size_t sgu = b.z_gate - b.s_gate, sd = b.z_down - b.s_down;
  std::memcpy(o + b.q_gate, q_gate, qgu);
  std::memcpy(o + b.q_up, q_up, qgu);
  std::memcpy(o + b.q_down, q_down, qd);
  std::memcpy(o + b.s_gate, s_gate, sgu);
  std::memcpy(o + b.z_gate, z_gate, sgu);
  std::memcpy(o + b.s_up, s_up, sgu);
  std::memcpy(o + b.z_up, z_up, sgu);
  std::memcpy(o + b.s_down, s_down, sd);
  std::memcpy(o + b.z_down, z_down, sd);
  return MOE_OK;
}

int moe_unpack_expert(const moe_expert_shape* s, const void* block,
                      uint8_t* q_gate, uint8_t* q_up, uint8_t* q_down,
                      uint16_t* s_gate, uint16_t* z_gate, uint16_t* s_up,
                      uint16_t* z_up, uint16_t* s_down, uint16_t* z_down) {
  moe::clear_error();
  if (!moe::valid_shape(s)) return moe::fail(MOE_ERR_SHAPE, "invalid expert shape");
  if (!q_gate || !q_up || !q_down || !s_gate || !z_gate || !s_up || !z_up ||
      !s_down || !z_down || !block)
    return moe::fail(MOE_ERR_ARG, "NULL array");
  const moe::BlockLayout b = moe::block_layout(s->hidden, s->inter, s->group);
  const uint8_t* i = static_cast<const uint8_t*>(block);
  const size_t qgu = b.q_up - b.q_gate, qd = b.s_gate - b.q_down;
  const size_t sgu = b.z_gate - b.s_gate, sd = b.z_down - b.s_down;
  std::memcpy(q_gate, i + b.q_gate, qgu);
  std::memcpy(q_up, i + b.q_up, qgu);
  std::memcpy(q_down, i + b.q_down, qd);
  std::memcpy(s_gate, i + b.s_gate, sgu);
  std::memcpy(z_gate, i + b.z_gate, sgu);
  std::memcpy(s_up, i + b.s_up, sgu);
  std::memcpy(z_up, i + b.z_up, sgu);
  std::memcpy(s_down, i + b.s_down, sd);
  std::memcpy(z_down, i + b.z_down, sd);
  return MOE_OK;
}

}  // extern "C"
