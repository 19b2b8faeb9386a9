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

int moe_expert_block_layout(const moe_expert_shape* s, moe_block_layout* out) {
  moe::clear_error();
  if (!out) return moe::fail(MOE_ERR_ARG, "out is NULL");
  if (!moe::valid_shape(s)) return moe::fail(MOE_ERR_SHAPE, "invalid expert shape");
  const moe::BlockLayout b = moe::block_layout(s->hidden, s->inter, s->group);
  out->total = b.total;
  out->d_offset = b.d_offset;
  out->gu_row_bytes = b.gu_row;
  out->d_row_bytes = b.d_row;
  out->gu_q_gate = b.gu_q_gate;
  out->gu_q_up = b.gu_q_up;
  out->gu_sz = b.gu_sz;
  out->d_q = b.d_q;
  out->d_sz = b.d_sz;
  return MOE_OK;
}

}  // extern "C"

namespace {
// Direction-agnostic row copy between the canonical arrays and a block.
template <bool kPack>
void copy_rows(const moe_expert_shape* s, uint8_t* blk, uint8_t* qg, uint8_t* qu, uint8_t* qd,
               uint8_t* sg, uint8_t* zg, uint8_t* su, uint8_t* zu, uint8_t* sd, uint8_t* zd) {
  const int H = s->hidden, I = s->inter, g = s->group;
  const moe::BlockLayout b = moe::block_layout(H, I, g);
  const size_t q_gu = (size_t)H / 2, s_gu = (size_t)(H / g) * 2;
  const size_t q_d = (size_t)I / 2, s_d = (size_t)(I / g) * 2;
  auto mv = [](uint8_t* blk_part, uint8_t* arr_part, size_t n) {
    if (kPack) std::memcpy(blk_part, arr_part, n);
    else std::memcpy(arr_part, blk_part, n);
  };
  (void)s_gu;
  (void)s_d;
  const int ggu = H / g, gd = I / g;
  if (kPack) std::memset(blk, 0, b.total);
  for (int n = 0; n < I; ++n) {
    uint8_t* row = blk + (size_t)n * b.gu_row;
    mv(row + b.gu_q_gate, qg + n * q_gu, q_gu);
    mv(row + b.gu_q_up, qu + n * q_gu, q_gu);
    for (int gi = 0; gi < ggu; ++gi) {
      uint8_t* quad = row + b.gu_sz + (size_t)gi * 8;
      const size_t e = ((size_t)n * ggu + gi) * 2;
      mv(quad + 0, sg + e, 2);
      mv(quad + 2, zg + e, 2);
      mv(quad + 4, su + e, 2);
      mv(quad + 6, zu + e, 2);
    }
  }
  for (int m = 0; m < H; ++m) {
    uint8_t* row = blk + b.d_offset + (size_t)m * b.d_row;
    mv(row + b.d_q, qd + m * q_d, q_d);
    for (int gi = 0; gi < gd; ++gi) {
      uint8_t* pr = row + b.d_sz + (size_t)gi * 4;
      const size_t e = ((size_t)m * gd + gi) * 2;
      mv(pr + 0, sd + e, 2);
      mv(pr + 2, zd + e, 2);
    }
  }
}
}  // namespace

extern "C" {

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
  auto c = [](const void* p) { return const_cast<uint8_t*>(static_cast<const uint8_t*>(p)); };
  copy_rows<true>(s, static_cast<uint8_t*>(block_out), c(q_gate), c(q_up), c(q_down), c(s_gate),
                  c(z_gate), c(s_up), c(z_up), c(s_down), c(z_down));
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
  auto c = [](void* p) { return static_cast<uint8_t*>(p); };
  copy_rows<false>(s, const_cast<uint8_t*>(static_cast<const uint8_t*>(block)), q_gate, q_up,
                   q_down, c(s_gate), c(z_gate), c(s_up), c(z_up), c(s_down), c(z_down));
  return MOE_OK;
}

}  // extern "C"
