// Non-routed FP16 SwiGLU FFN ("Horizon RunMap -- Prévia Técnica",
// "03 / Arquitetura" and "08 / Comportamento do modelo": the parts outside
// the routed experts keep FP16 weights):
//   y = W_d (silu(W_g x) * (W_u x)),  W_g, W_u [Is][H], W_d [H][Is], FP16.
//
// Two tensor-core GEMM kernels; both take the weight rows as the 128-row MMA
// operand and the tokens as the N operand, both operands brought by TMA in
// the 128-byte-swizzled K-major layout tcgen05.mma reads, FP32 accumulation
// in tensor memory:
//   1. gate/up: per (128 rows of Is, 256 tokens) a gate and an up
//      accumulator; the epilogue forms h = silu(gate) * up, FP16 [T][Is];
//   2. down: per (128 rows of H, 128 tokens) two accumulators over the even
//      and odd 16-element K slices, added in the epilogue; y stored as FP16.
#include <algorithm>
#include <mutex>

#include "common.h"
#include "device.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int kGuN = 256;  // tokens per gate/up tile (two 256-column accumulators fill tensor memory)
constexpr int kDnN = 128;  // tokens per down tile (two K-slice accumulators)
// Warp roles: 0 TMA, 1 TMEM + MMA issue (accumulator 0), 2 idle, 3 MMA issue
// (accumulator 1), 4..11 epilogue. One thread issues a tcgen05.mma about every
// 120 cycles, so two issuing threads with an accumulator each keep the tensor
// cores busier.
constexpr int kThreads = 384;
constexpr uint32_t kWTile = BM * BK * 2;  // 16 KB weight tile
// gate/up stage: W_g tile | W_u tile | x tile (256 tokens); down stage: W_d tile | h tile (128 tokens).
constexpr int kGuStages = 3, kDnStages = 6;
constexpr uint32_t kGuStage = 2 * kWTile + kGuN * BK * 2, kDnStage = kWTile + kDnN * BK * 2;
constexpr size_t kGuSmem = (size_t)kGuStages * kGuStage + 2048;
constexpr size_t kDnSmem = (size_t)kDnStages * kDnStage + 2048;
static_assert(kGuStage % 1024 == 0 && kDnStage % 1024 == 0, "stage alignment");

struct SharedParams {
  int rows;  // Is (gate/up) or H (down)
  int K;     // H (gate/up) or Is (down)
  int T;
  __half* out;  // h [T][Is] or y [T][H]
  int32_t* flags;
};

// Producer: per K step the weight tile(s) at row0 and the token tile at tok0.
// The whole warp runs the loop and one elected lane issues the copies.
template <int NW, int STAGES>
__device__ __forceinline__ void produce_tiles(const tc::Ctrl& c, uint8_t* sm, uint32_t stage_bytes,
                                              uint32_t tok_bytes, const CUtensorMap* w0, const CUtensorMap* w1,
                                              const CUtensorMap* tok, int row0, int tok0, int KT, int32_t* flags) {
  const int lane = threadIdx.x & 31;
  int issued = 0;
  for (int kt = 0; kt < KT; ++kt) {
    const int s = kt % STAGES;
    if (kt >= STAGES && !tc::bar_wait_warp(&c.empty[s], ((kt / STAGES) - 1) & 1)) {
      if (lane == 0) tc::set_abort(c, flags);
      break;
    }
    if (__any_sync(0xffffffffu, tc::aborted(c))) break;
    uint8_t* st = sm + (size_t)s * stage_bytes;
    const int k0 = kt * BK;
    if (tc::elect_one()) {
      tc::bar_expect_tx(&c.tma_full[s], NW * kWTile + tok_bytes);
      tc::tma_load_2d(st, w0, k0, row0, &c.tma_full[s]);
      if (NW == 2) tc::tma_load_2d(st + kWTile, w1, k0, row0, &c.tma_full[s]);
      tc::tma_load_2d(st + NW * kWTile, tok, k0, tok0, &c.tma_full[s]);
    }
    __syncwarp();
    issued = kt + 1;
  }
  if (lane == 0 && tc::aborted(c)) tc::drain_loads(c, STAGES, issued);
}

__device__ __forceinline__ void setup_bars(const tc::Ctrl& c, int stages) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::bar_init(&c.tma_full[s], 1);
      tc::bar_init(&c.empty[s], 2);  // one commit per issuing thread
    }
    tc::bar_init(c.acc_full, 2);
    *c.abort = 0;
    tc::bar_init_fence();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    shared_gateup_kernel(const __grid_constant__ CUtensorMap map_wg, const __grid_constant__ CUtensorMap map_wu,
                         const __grid_constant__ CUtensorMap map_x, const SharedParams a) {
  const int row0 = blockIdx.x * BM, tok0 = blockIdx.y * kGuN;
  const int n = min(kGuN, a.T - tok0);
  const int nmma = (n + 15) & ~15;
  const int KT = a.K / BK;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = tc::align1024(smraw);
  const tc::Ctrl c = tc::ctrl_at(sm + (size_t)kGuStages * kGuStage, kGuStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::tma_prefetch_desc(&map_wg);
    tc::tma_prefetch_desc(&map_wu);
    tc::tma_prefetch_desc(&map_x);
  }
  setup_bars(c, kGuStages);
  if (warp == 1) tc::tmem_alloc(c.tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *c.tmem_slot;
  if (warp == 0) {
    produce_tiles<2, kGuStages>(c, sm, kGuStage, kGuN * BK * 2, &map_wg, &map_wu, &map_x, row0, tok0, KT, a.flags);
  } else if (warp == 1 || warp == 3) {
    // Issuer p: the gate (p = 0) or up (p = 1) projection. The whole warp
    // runs the loop, one elected lane issues.
    const int p = warp == 1 ? 0 : 1;
    const uint32_t idesc = tc::idesc_f16(BM, nmma);
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % kGuStages;
      if (!tc::bar_wait_warp(&c.tma_full[s], (kt / kGuStages) & 1)) {
        if (lane == 0) tc::set_abort(c, a.flags);
        break;
      }
      if (__any_sync(0xffffffffu, tc::aborted(c))) break;
      tc::tc_fence_after();
      const uint32_t base = tc::smem_addr(sm + (size_t)s * kGuStage);
      if (tc::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma_f16(tmem + p * kGuN, tc::sw128_desc(base + p * kWTile + kk * 32),
                      tc::sw128_desc(base + 2 * kWTile + kk * 32), idesc, kt > 0 || kk > 0);
        tc::mma_commit(&c.empty[s]);
      }
      __syncwarp();
    }
    if (tc::elect_one()) tc::mma_commit(c.acc_full);
    __syncwarp();
  } else if (warp >= 4) {
    const bool ok = tc::bar_wait(c.acc_full, 0);
    if (!ok) tc::set_abort(c, a.flags);
    tc::tc_fence_after();
    const int q4 = warp & 3, chalf = (warp - 4) >> 2;
    const int row = row0 + 32 * q4 + lane;
    const bool live = ok && !tc::aborted(c) && row < a.rows;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    for (int c0 = chalf * (kGuN / 2); c0 < chalf * (kGuN / 2) + kGuN / 2 && c0 < nmma; c0 += 16) {
      float gv[16], uv[16];
      tc::tmem_ld16(tl + (uint32_t)c0, gv);
      tc::tmem_ld16(tl + (uint32_t)(kGuN + c0), uv);
      tc::tmem_ld_wait();
      if (live) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < n) a.out[(size_t)(tok0 + c0 + j) * a.rows + row] = __float2half_rn(silu_fast(gv[j]) * uv[j]);
      }
    }
  }
  tc::gemm_teardown(tmem, 512);
}

__global__ void __launch_bounds__(kThreads, 1)
    shared_down_kernel(const __grid_constant__ CUtensorMap map_wd, const __grid_constant__ CUtensorMap map_h,
                       const SharedParams a) {
  const int row0 = blockIdx.x * BM, tok0 = blockIdx.y * kDnN;
  const int n = min(kDnN, a.T - tok0);
  const int nmma = (n + 15) & ~15;
  const int KT = a.K / BK;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = tc::align1024(smraw);
  const tc::Ctrl c = tc::ctrl_at(sm + (size_t)kDnStages * kDnStage, kDnStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::tma_prefetch_desc(&map_wd);
    tc::tma_prefetch_desc(&map_h);
  }
  setup_bars(c, kDnStages);
  if (warp == 1) tc::tmem_alloc(c.tmem_slot, 2 * kDnN);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *c.tmem_slot;
  if (warp == 0) {
    produce_tiles<1, kDnStages>(c, sm, kDnStage, kDnN * BK * 2, &map_wd, nullptr, &map_h, row0, tok0, KT, a.flags);
  } else if (warp == 1 || warp == 3) {
    // Issuer p: the K slices kk = p, p + 2 of every step, into accumulator p.
    // The whole warp runs the loop, one elected lane issues.
    const int p = warp == 1 ? 0 : 1;
    const uint32_t idesc = tc::idesc_f16(BM, nmma);
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % kDnStages;
      if (!tc::bar_wait_warp(&c.tma_full[s], (kt / kDnStages) & 1)) {
        if (lane == 0) tc::set_abort(c, a.flags);
        break;
      }
      if (__any_sync(0xffffffffu, tc::aborted(c))) break;
      tc::tc_fence_after();
      const uint32_t base = tc::smem_addr(sm + (size_t)s * kDnStage);
      if (tc::elect_one()) {
#pragma unroll
        for (int kk = p; kk < BK / 16; kk += 2)
          tc::mma_f16(tmem + p * kDnN, tc::sw128_desc(base + kk * 32), tc::sw128_desc(base + kWTile + kk * 32), idesc,
                      kt > 0 || kk > p);
        tc::mma_commit(&c.empty[s]);
      }
      __syncwarp();
    }
    if (tc::elect_one()) tc::mma_commit(c.acc_full);
    __syncwarp();
  } else if (warp >= 4) {
    const bool ok = tc::bar_wait(c.acc_full, 0);
    if (!ok) tc::set_abort(c, a.flags);
    tc::tc_fence_after();
    const int q4 = warp & 3, chalf = (warp - 4) >> 2;
    const int row = row0 + 32 * q4 + lane;
    const bool live = ok && !tc::aborted(c) && row < a.rows;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    for (int c0 = chalf * (kDnN / 2); c0 < chalf * (kDnN / 2) + kDnN / 2 && c0 < nmma; c0 += 16) {
      float dv[16], ev[16];
      tc::tmem_ld16(tl + (uint32_t)c0, dv);
      tc::tmem_ld16(tl + (uint32_t)(kDnN + c0), ev);
      tc::tmem_ld_wait();
      if (live) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < n) a.out[(size_t)(tok0 + c0 + j) * a.rows + row] = __float2half_rn(dv[j] + ev[j]);
      }
    }
  }
  tc::gemm_teardown(tmem, 2 * kDnN);
}

// Per device: the kernels' shared-memory attribute has been set.
std::mutex g_attr_mutex;
bool g_attr_set[kMaxDevices] = {};

int fp16_map(CUtensorMap* m, const void* base, int inner, int outer, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)inner, (uint64_t)outer};
  const uint64_t str[1] = {(uint64_t)inner * 2};
  const uint32_t box[2] = {BK, (uint32_t)box_rows};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_shared_workspace_bytes(int T, int H, int Is) {
  if (T < 0 || H <= 0 || Is <= 0) return 0;
  return moe::kWorkspaceHeader + (size_t)T * Is * 2;
}

extern "C" int moe_shared_forward(const void* x, int T, int H, int Is, const void* wg,
                                  const void* wu, const void* wd, void* y, void* ws,
                                  size_t ws_bytes, void* stream) {
  moe::NvtxRange nvtx_range("moe_shared_forward");
  moe::clear_error();
  if (T < 0 || H <= 0 || Is <= 0 || H % 64 || Is % 64 || H > 65536 || Is > 65536)
    return moe::fail(MOE_ERR_ARG, "moe_shared_forward: need H, Is positive multiples of 64 (H=%d Is=%d T=%d)", H,
                     Is, T);
  if (T == 0) return MOE_OK;
  if (!x || !wg || !wu || !wd || !y || !ws) return moe::fail(MOE_ERR_ARG, "moe_shared_forward: NULL pointer");
  const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(wg) |
                       reinterpret_cast<uintptr_t>(wu) | reinterpret_cast<uintptr_t>(wd) |
                       reinterpret_cast<uintptr_t>(y);
  if (al % 16 || reinterpret_cast<uintptr_t>(ws) % 256)
    return moe::fail(MOE_ERR_ARG, "moe_shared_forward: x, weights, y 16-byte and workspace 256-byte aligned");
  const size_t need = moe_shared_workspace_bytes(T, H, Is);
  if (ws_bytes < need)
    return moe::fail(MOE_ERR_CAPACITY, "moe_shared_forward: workspace %zu < %zu bytes", ws_bytes, need);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  int32_t* flags = reinterpret_cast<int32_t*>(w8);
  __half* h = reinterpret_cast<__half*>(w8 + moe::kWorkspaceHeader);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap m_wg, m_wu, m_x, m_wd, m_h;
  int rc;
  if ((rc = moe::fp16_map(&m_wg, wg, H, Is, moe::BM)) != MOE_OK) return rc;
  if ((rc = moe::fp16_map(&m_wu, wu, H, Is, moe::BM)) != MOE_OK) return rc;
  if ((rc = moe::fp16_map(&m_x, x, H, T, moe::kGuN)) != MOE_OK) return rc;
  if ((rc = moe::fp16_map(&m_wd, wd, Is, H, moe::BM)) != MOE_OK) return rc;
  if ((rc = moe::fp16_map(&m_h, h, Is, T, moe::kDnN)) != MOE_OK) return rc;
  int dev = 0, n_sm = 0;
  if ((rc = moe::current_device_sms(&dev, &n_sm)) != MOE_OK) return rc;
  {
    std::lock_guard<std::mutex> lock(moe::g_attr_mutex);
    if (!moe::g_attr_set[dev]) {
      MOE_CUDA_TRY(cudaFuncSetAttribute(moe::shared_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)moe::kGuSmem));
      MOE_CUDA_TRY(cudaFuncSetAttribute(moe::shared_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)moe::kDnSmem));
      moe::g_attr_set[dev] = true;
    }
  }
  moe::SharedParams p;
  p.T = T;
  p.flags = flags;
  p.rows = Is;
  p.K = H;
  p.out = h;
  moe::shared_gateup_kernel<<<dim3((Is + moe::BM - 1) / moe::BM, (T + moe::kGuN - 1) / moe::kGuN), moe::kThreads,
                              moe::kGuSmem, st>>>(m_wg, m_wu, m_x, p);
  if ((rc = moe::check_launch("shared gate/up GEMM")) != MOE_OK) return rc;
  p.rows = H;
  p.K = Is;
  p.out = static_cast<__half*>(y);
  moe::shared_down_kernel<<<dim3((H + moe::BM - 1) / moe::BM, (T + moe::kDnN - 1) / moe::kDnN), moe::kThreads,
                            moe::kDnSmem, st>>>(m_wd, m_h, p);
  return moe::check_launch("shared down GEMM");
}
