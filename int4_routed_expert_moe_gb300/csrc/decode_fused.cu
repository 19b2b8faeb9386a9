// Decode path, fused: one persistent kernel per routed layer.
//
// "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura" and
// "08 / Comportamento do modelo": the expert kernel reads compact INT4 codes
// and FP16 scales, converts them inside the kernel (no expanded expert is
// kept) and works with FP16 activations and FP32 accumulation.
//
// Work split (G blocks, one per SM, all resident at once):
//   * block c owns gate/up rows n in [c*I/G, (c+1)*I/G) of every (token,
//     choice) pair p, and output rows m in [c*H/G, (c+1)*H/G) of y.
//   * A producer warp streams, pair after pair, the block's slice of expert
//     ids[p]'s block (gate/up code rows + their scales/zeros, down code rows +
//     scales/zeros) into a ring of shared-memory stages with bulk async
//     copies (cp.async.bulk + mbarrier transaction counts). For one decode
//     token the whole layer slice (~176 KB per SM) is requested at once.
//   * Consumer warps compute h[p][n] = silu(g) * u for the block's rows as a
//     stage lands, store h (FP16, the explicit rounding point) to the
//     workspace and publish the row count on a per-pair counter (release).
//   * The down projection of pair p waits (acquire, bounded) until all I rows
//     of h[p] are published, then adds w[p] * W_d h[p] for the block's output
//     rows, using the stage's down rows. Pair p's down work runs after pair
//     p+1's gate/up work, so it overlaps the stream of later pairs.
//   * The last block to finish resets the counters, leaving the workspace
//     ready for the next call.
// Waits are bounded: on expiry the block sets bit 2 of the workspace error
// word and carries on, so a broken invariant gives a wrong result and an
// error flag, never a hang.
#include "common.h"
#include "device.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + producer warp
constexpr int kMaxStages = 8;
constexpr unsigned kSpinLimit = 1u << 20;             // bounded polling of waits

// ---- PTX wrappers: mbarrier, bulk copies, acquire/release -----------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase; returns false on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (unsigned i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
// Named barrier over the consumer warps only (the producer never joins).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// ---- static layout of one shared-memory stage -----------------------------
struct StageLayout {
  // byte offsets inside a stage
  uint32_t qg, qu, sg, zg, su, zu, qd, sd, zd, bytes;
  uint32_t sgu_row_bytes, sd_row_bytes;
  uint32_t span_gu, span_d;  // bytes copied per scale/zero slice (16-aligned superset)
};

__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline StageLayout stage_layout(int H, int I, int g, int rgu, int rdn) {
  StageLayout L;
  L.sgu_row_bytes = (uint32_t)(H / g) * 2u;
  L.sd_row_bytes = (uint32_t)(I / g) * 2u;
  // A slice of rows r0..r0+R of a scale array is copied as the 16-aligned
  // superset [align_down(start), align_up(end)), at most R*row + 32 bytes.
  L.span_gu = align16((uint32_t)rgu * L.sgu_row_bytes + 32u);
  L.span_d = align16((uint32_t)rdn * L.sd_row_bytes + 32u);
  uint32_t o = 0;
  L.qg = o; o += align16((uint32_t)rgu * (H / 2));
  L.qu = o; o += align16((uint32_t)rgu * (H / 2));
  L.qd = o; o += align16((uint32_t)rdn * (I / 2));
  L.sg = o; o += L.span_gu;
  L.zg = o; o += L.span_gu;
  L.su = o; o += L.span_gu;
  L.zu = o; o += L.span_gu;
  L.sd = o; o += L.span_d;
  L.zd = o; o += L.span_d;
  L.bytes = align16(o);
  return L;
}

struct FusedParams {
  const __half* x;
  const int32_t* ids;
  const float* wts;
  const uint8_t* pool;
  unsigned long long block_bytes;
  BlockOffsets off;
  const int32_t* slot_of;
  const __half* y_shared;
  __half* y;
  int32_t* flags;      // workspace error word
  int32_t* exit_cnt;   // workspace: blocks finished
  int32_t* pair_cnt;   // workspace: [P] rows of h published per pair
  __half* hbuf;        // workspace: [P][I]
  int H, I, g, T, k, E, n_slots, P, G, stages;
  StageLayout st;
  uint32_t x_off, h_off, acc_off, bar_off;  // shared-memory carve-up
};

__device__ __forceinline__ const uint8_t* resolve(const FusedParams& a, int p) {
  const int e = a.ids[p];
  if (e < 0 || e >= a.E) return nullptr;
  const int s = a.slot_of[e];
  if (s < 0 || s >= a.n_slots) return nullptr;
  return a.pool + (size_t)s * a.block_bytes;
}

// Rows [r0, r1) of a scale/zero array (row_bytes each) are copied as the
// 16-byte aligned superset [start, start + bytes); row r0 sits at `skip`.
struct ScaleSpan {
  uint32_t start, bytes, skip;
};
__device__ __forceinline__ ScaleSpan scale_span(int r0, int r1, uint32_t row_bytes) {
  ScaleSpan sp;
  const uint32_t s0 = (uint32_t)r0 * row_bytes, s1 = (uint32_t)r1 * row_bytes;
  sp.start = s0 & ~15u;
  sp.bytes = r1 > r0 ? ((s1 + 15u) & ~15u) - sp.start : 0u;
  sp.skip = s0 - sp.start;
  return sp;
}

__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(const FusedParams a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int n0 = (int)(((long long)c * a.I) / a.G), n1 = (int)(((long long)(c + 1) * a.I) / a.G);
  const int m0 = (int)(((long long)c * a.H) / a.G), m1 = (int)(((long long)(c + 1) * a.H) / a.G);
  const int rgu = n1 - n0, rdn = m1 - m0;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + a.bar_off);
  uint64_t* empty = full + kMaxStages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // Everything below reads what earlier kernels wrote (ids, x, the pool).
  griddep_wait();
  griddep_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      const StageLayout& L = a.st;
      const uint32_t qgu_bytes = (uint32_t)rgu * (a.H / 2), qd_bytes = (uint32_t)rdn * (a.I / 2);
      const ScaleSpan sg = scale_span(n0, n1, L.sgu_row_bytes);
      const ScaleSpan sd = scale_span(m0, m1, L.sd_row_bytes);
      const uint32_t total = (rgu > 0 ? 2 * qgu_bytes + 4 * sg.bytes : 0u) +
                             (rdn > 0 ? qd_bytes + 2 * sd.bytes : 0u);
      for (int p = 0; p < a.P; ++p) {
        const int s = p % a.stages;
        if (p >= a.stages) {
          if (!mbar_wait(&empty[s], ((p / a.stages) - 1) & 1)) atomicOr(a.flags, 4);
        }
        uint8_t* stg = sm + (size_t)s * L.bytes;
        const uint8_t* blk = resolve(a, p);
        if (!blk) {
          mbar_arrive_expect_tx(&full[s], 0);
          continue;
        }
        mbar_arrive_expect_tx(&full[s], total);
        if (rgu > 0) {
          bulk_g2s(stg + L.qg, blk + a.off.q_gate + (size_t)n0 * (a.H / 2), qgu_bytes, &full[s]);
          bulk_g2s(stg + L.qu, blk + a.off.q_up + (size_t)n0 * (a.H / 2), qgu_bytes, &full[s]);
          if (sg.bytes) {
            bulk_g2s(stg + L.sg, blk + a.off.s_gate + sg.start, sg.bytes, &full[s]);
            bulk_g2s(stg + L.zg, blk + a.off.z_gate + sg.start, sg.bytes, &full[s]);
            bulk_g2s(stg + L.su, blk + a.off.s_up + sg.start, sg.bytes, &full[s]);
            bulk_g2s(stg + L.zu, blk + a.off.z_up + sg.start, sg.bytes, &full[s]);
          }
        }
        if (rdn > 0) {
          bulk_g2s(stg + L.qd, blk + a.off.q_down + (size_t)m0 * (a.I / 2), qd_bytes, &full[s]);
          if (sd.bytes) {
            bulk_g2s(stg + L.sd, blk + a.off.s_down + sd.start, sd.bytes, &full[s]);
            bulk_g2s(stg + L.zd, blk + a.off.z_down + sd.start, sd.bytes, &full[s]);
          }
        }
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int tid = threadIdx.x;  // 0 .. kConsumerWarps*32-1
  __half* xs = reinterpret_cast<__half*>(sm + a.x_off);           // [H] pair order
  float* xsum = reinterpret_cast<float*>(sm + a.x_off + a.H * 2);  // [H/32]
  __half* hs = reinterpret_cast<__half*>(sm + a.h_off);           // [I] pair order
  float* hsum = reinterpret_cast<float*>(sm + a.h_off + a.I * 2);  // [I/32]
  float* acc = reinterpret_cast<float*>(sm + a.acc_off);          // [T][rdn]
  for (int i = tid; i < a.T * rdn; i += kConsumerWarps * 32) acc[i] = 0.0f;
  int cur_t = -1;
  bool timed_out = false;

  auto stage_vec = [&](const __half* src, int n, __half* dst, float* sums, bool coherent) {
    const int nb = n / 8;
    for (int base = 0; base < nb; base += kConsumerWarps * 32) {
      const int b = base + tid;
      float s = 0.0f;
      if (b < nb) {
        const uint4 v = coherent ? ld_cg_v4(src + 8 * b) : *reinterpret_cast<const uint4*>(src + 8 * b);
        __half e[8];
        *reinterpret_cast<uint4*>(e) = v;
        store_perm8(dst + 8 * b, e);
#pragma unroll
        for (int i = 0; i < 8; ++i) s += __half2float(e[i]);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (b < nb && (b & 3) == 0) sums[b >> 2] = s;
    }
  };

  // Down projection of pair q from stage q % stages.
  auto down_pair = [&](int q) {
    const int s = q % a.stages;
    const uint8_t* blk = resolve(a, q);
    if (blk && rdn > 0) {
      if (tid == 0) {
        unsigned i = 0;
        while (ld_acquire(a.pair_cnt + q) < a.I) {
          if (++i > kSpinLimit) {
            atomicOr(a.flags, 4);
            timed_out = true;
            break;
          }
          __nanosleep(32);
        }
      }
      consumers_sync();
      stage_vec(a.hbuf + (size_t)q * a.I, a.I, hs, hsum, true);
      consumers_sync();
      const uint8_t* stg = sm + (size_t)s * a.st.bytes;
      const uint32_t skip = scale_span(m0, m1, a.st.sd_row_bytes).skip;
      const __half* sd = reinterpret_cast<const __half*>(stg + a.st.sd + skip);
      const __half* zd = reinterpret_cast<const __half*>(stg + a.st.zd + skip);
      const int t = q / a.k;
      const float wq = a.wts[q];
      const int nch = a.I / 32, gpr = a.I / a.g;
      for (int r = warp; r < rdn; r += kConsumerWarps) {
        const uint8_t* row = stg + a.st.qd + (size_t)r * (a.I / 2);
        float part = 0.0f;
        for (int cc = lane; cc < nch; cc += 32) {
          const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * cc);
          const float d = dot32_codes(w, reinterpret_cast<const half2*>(hs + 32 * cc));
          const int gi = (32 * cc) / a.g;
          part += __half2float(sd[r * gpr + gi]) * (d - __half2float(zd[r * gpr + gi]) * hsum[cc]);
        }
        part = warp_sum(part);
        if (lane == 0) acc[t * rdn + r] += wq * part;
      }
      consumers_sync();  // hs is reused by the next pair
    }
    if (tid == 0) mbar_arrive(&empty[s]);
  };

  for (int p = 0; p < a.P; ++p) {
    const int s = p % a.stages;
    const int t = p / a.k;
    if (t != cur_t) {
      stage_vec(a.x + (size_t)t * a.H, a.H, xs, xsum, false);
      cur_t = t;
    }
    if (!mbar_wait(&full[s], (p / a.stages) & 1)) {
      if (tid == 0) atomicOr(a.flags, 4);
      timed_out = true;
    }
    consumers_sync();  // x staged, stage visible to all consumers
    const uint8_t* blk = resolve(a, p);
    if (rgu > 0) {
      const uint8_t* stg = sm + (size_t)s * a.st.bytes;
      const int gpr = a.H / a.g, nch = a.H / 32;
      const uint32_t skip = scale_span(n0, n1, a.st.sgu_row_bytes).skip;
      const __half* sg = reinterpret_cast<const __half*>(stg + a.st.sg + skip);
      const __half* zg = reinterpret_cast<const __half*>(stg + a.st.zg + skip);
      const __half* su = reinterpret_cast<const __half*>(stg + a.st.su + skip);
      const __half* zu = reinterpret_cast<const __half*>(stg + a.st.zu + skip);
      for (int r = warp; r < rgu; r += kConsumerWarps) {
        float hv = 0.0f;
        if (blk) {
          const uint8_t* rg = stg + a.st.qg + (size_t)r * (a.H / 2);
          const uint8_t* ru = stg + a.st.qu + (size_t)r * (a.H / 2);
          float ag = 0.0f, au = 0.0f;
          for (int cc = lane; cc < nch; cc += 32) {
            const uint4 wg = *reinterpret_cast<const uint4*>(rg + 16 * cc);
            const uint4 wu = *reinterpret_cast<const uint4*>(ru + 16 * cc);
            const half2* xp = reinterpret_cast<const half2*>(xs + 32 * cc);
            const float dg = dot32_codes(wg, xp);
            const float du = dot32_codes(wu, xp);
            const int gi = (32 * cc) / a.g;
            const float xsm = xsum[cc];
            ag += __half2float(sg[r * gpr + gi]) * (dg - __half2float(zg[r * gpr + gi]) * xsm);
            au += __half2float(su[r * gpr + gi]) * (du - __half2float(zu[r * gpr + gi]) * xsm);
          }
          ag = warp_sum(ag);
          au = warp_sum(au);
          hv = silu_f(ag) * au;
        }
        if (lane == 0) {
          a.hbuf[(size_t)p * a.I + n0 + r] = __float2half_rn(hv);
          __threadfence();  // each writer orders its h before the block's publish
        }
      }
      consumers_sync();  // all rows of this pair stored
      if (tid == 0) {
        __threadfence();
        atomicAdd(a.pair_cnt + p, rgu);
      }
    }
    if (p >= 1) down_pair(p - 1);
  }
  if (a.P >= 1) down_pair(a.P - 1);
  consumers_sync();
  // Output rows of this block.
  for (int i = tid; i < a.T * rdn; i += kConsumerWarps * 32) {
    const int t = i / rdn, r = i - t * rdn;
    float v = acc[i];
    if (a.y_shared) v += __half2float(a.y_shared[(size_t)t * a.H + m0 + r]);
    a.y[(size_t)t * a.H + m0 + r] = __float2half_rn(v);
  }
  // Last block out resets the pair counters for the next call.
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(a.exit_cnt, 1);
    if (prev == a.G - 1) {
      for (int p = 0; p < a.P; ++p) a.pair_cnt[p] = 0;
      *a.exit_cnt = 0;
      __threadfence();
    }
  }
  (void)timed_out;
}

int g_num_sms = 0;

}  // namespace

// Workspace of the fused decode path: header | pair counters | h [P][I] fp16.
static size_t fused_counter_off() { return kWorkspaceHeader; }
static size_t fused_h_off(int P) { return kWorkspaceHeader + (((size_t)P * 4 + 255) / 256) * 256; }

size_t fused_workspace_bytes(int H, int I, int T, int k) {
  (void)H;
  const int P = T * k;
  return fused_h_off(P) + (size_t)P * I * 2;
}

int fused_forward(const ForwardArgs& fa) {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  }
  FusedParams a;
  a.H = fa.H; a.I = fa.I; a.g = fa.g; a.T = fa.T; a.k = fa.k; a.E = fa.E; a.n_slots = fa.n_slots;
  a.P = fa.T * fa.k;
  a.G = g_num_sms;
  a.x = fa.x; a.ids = fa.ids; a.wts = fa.weights; a.pool = fa.pool; a.block_bytes = fa.block_bytes;
  a.off = fa.off; a.slot_of = fa.slot_of; a.y_shared = fa.y_shared; a.y = fa.y;
  uint8_t* ws = static_cast<uint8_t*>(fa.ws);
  a.flags = reinterpret_cast<int32_t*>(ws);
  a.exit_cnt = reinterpret_cast<int32_t*>(ws + 4);
  a.pair_cnt = reinterpret_cast<int32_t*>(ws + fused_counter_off());
  a.hbuf = reinterpret_cast<__half*>(ws + fused_h_off(a.P));
  const int rgu_max = (a.I + a.G - 1) / a.G, rdn_max = (a.H + a.G - 1) / a.G;
  a.st = stage_layout(a.H, a.I, a.g, rgu_max, rdn_max);
  const size_t fixed = (size_t)a.H * 2 + (size_t)(a.H / 32) * 4   // x
                       + (size_t)a.I * 2 + (size_t)(a.I / 32) * 4  // h
                       + (size_t)a.T * rdn_max * 4                 // acc
                       + 2 * kMaxStages * 8 + 256;
  const size_t budget = 220 * 1024;
  if (fixed + 2 * (size_t)a.st.bytes > budget)
    return fail(MOE_ERR_UNSUPPORTED, "fused decode: shapes need %zu bytes of shared memory",
                fixed + 2 * (size_t)a.st.bytes);
  a.stages = (int)std::min<size_t>(kMaxStages, (budget - fixed) / a.st.bytes);
  size_t o = (size_t)a.stages * a.st.bytes;
  a.x_off = (uint32_t)o; o += align16((uint32_t)(a.H * 2 + (a.H / 32) * 4));
  a.h_off = (uint32_t)o; o += align16((uint32_t)(a.I * 2 + (a.I / 32) * 4));
  a.acc_off = (uint32_t)o; o += align16((uint32_t)(a.T * rdn_max * 4));
  a.bar_off = (uint32_t)o; o += 2 * kMaxStages * 8;
  const size_t smem = o;
  static size_t s_attr = 0;
  if (smem > s_attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "fused decode smem attr: %s", cudaGetErrorString(e));
    s_attr = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = fa.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_fused_kernel, a);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "fused decode launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace moe
