// Decode path of the routed expert FFN: fused INT4 dequant-GEMV kernels.
//
// "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura" and
// "08 / Comportamento do modelo": the expert kernel reads compact INT4
// weights and FP16 scales, converts them inside the kernel (no expanded
// expert is kept) and uses FP16 activations with FP32 accumulation.
//
//   gateup_gemv_kernel: h[p][n] = silu(W_g x_t)[n] * (W_u x_t)[n] for every
//     (token, choice) pair p = t*k + j, read from expert ids[p]'s block.
//   down_gemv_kernel:   y[t][m] = sum_j w[t][j] * (W_d h_p)[m] (+ y_shared),
//     the top-k weighted combine fused into the down projection.
//
// Zero points: sum_c (q_c - z) s x_c = s * (sum_c q_c x_c - z * sum_c x_c)
// per 32-element chunk (a chunk never straddles a group since g % 32 == 0),
// with the chunk sums of x precomputed once per block. The products q_c x_c
// are FP16 (sums of at most 8 per lane) on the activations scaled per chunk
// by a power of two (dot16_scaled), so no product leaves the FP16 range
// whatever the activations' magnitude.
#include "common.h"
#include "device.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarps = 8;  // warps per block of both kernels

// Resolve the block of expert e, or NULL (setting the flag word) if it is
// not usable. e == -1 means "no expert" and is silent. An expert without a
// slot (slot_of[e] < 0) is read in place from `host` ([E][block], page-locked
// host memory mapped into the device's address space) when that is given.
__device__ __forceinline__ const uint8_t* expert_block(
    int e, int E, const int32_t* __restrict__ slot_of, int n_slots,
    const uint8_t* __restrict__ pool, size_t block_bytes, const uint8_t* __restrict__ host,
    int32_t* flags) {
  if (e < 0 || e >= E) {
    if (e != -1 && flags) atomicOr(flags, 2);
    return nullptr;
  }
  const int s = slot_of[e];
  if (s >= 0 && s < n_slots) return pool + (size_t)s * block_bytes;
  if (s < 0 && host) return host + (size_t)e * block_bytes;
  if (flags) atomicOr(flags, 1);
  return nullptr;
}

// Activations of one 8-element piece as the scaled pairs of dot16_scaled:
// the 4 threads of a 32-element chunk are adjacent lanes; they combine the
// chunk's largest magnitude and sum with shuffles, scale the chunk by the
// power of two 2^s that keeps every product an FP16 normal (chunk_shift),
// and the chunk keeps its FP32 sum (xsum) and the factor back 2^(24-s)
// (xback). All threads run the same number of iterations so the shuffles
// see full warps.
__device__ __forceinline__ void stage_piece(const float (&v)[8], bool valid, int b, __half* xs, float* xsum,
                                            float* xback) {
  float s = 0.0f, amax = 0.0f;
  if (valid) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s += v[i];
      amax = fmaxf(amax, fabsf(v[i]));
    }
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  if (valid) {
    const int sh = chunk_shift(amax);
    scaled_perm8(v, sh, reinterpret_cast<half2*>(xs + 8 * b));
    if ((b & 3) == 0) {
      xsum[b >> 2] = s;
      xback[b >> 2] = pow2f(24 - sh);
    }
  }
}

// Load FP16 activations [n] into shared memory as scaled pairs.
__device__ __forceinline__ void stage_activations(const __half* __restrict__ src, int n, __half* xs,
                                                  float* xsum, float* xback) {
  const int nb = n / 8;
  for (int base = 0; base < nb; base += blockDim.x) {
    const int b = base + threadIdx.x;
    float v[8];
    if (b < nb) {
      const uint4 raw = *reinterpret_cast<const uint4*>(src + 8 * b);
      const __half* a = reinterpret_cast<const __half*>(&raw);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __half2float(a[i]);
    }
    stage_piece(v, b < nb, b, xs, xsum, xback);
  }
}

// Same for FP32 intermediate values: round to FP16 first (the explicit
// rounding point before the down projection).
__device__ __forceinline__ void stage_rounded(const float* __restrict__ src, int n, __half* xs, float* xsum,
                                              float* xback) {
  const int nb = n / 8;
  for (int base = 0; base < nb; base += blockDim.x) {
    const int b = base + threadIdx.x;
    float v[8];
    if (b < nb) {
      const float4 v0 = *reinterpret_cast<const float4*>(src + 8 * b);
      const float4 v1 = *reinterpret_cast<const float4*>(src + 8 * b + 4);
      const float f[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __half2float(__float2half_rn(f[i]));
    }
    stage_piece(v, b < nb, b, xs, xsum, xback);
  }
}

// Dot of the 32 codes of a 16-byte chunk with the chunk's scaled pairs.
__device__ __forceinline__ float dot32_scaled(const uint4& w, const half2* xp, float back) {
  return (dot16_scaled(w.x, w.y, xp) + dot16_scaled(w.z, w.w, xp + 8)) * back;
}

// grid (ceil(I / kWarps), P); one warp per row n, gate and up rows together.
// NIT = iterations of the lane loop over 16-byte chunks (H / 1024, >= 1).
template <int NIT>
__global__ void __launch_bounds__(kWarps * 32) gateup_gemv_kernel(
    const __half* __restrict__ x, const int32_t* __restrict__ ids, int k, int E,
    const uint8_t* __restrict__ pool, size_t block_bytes,
    const int32_t* __restrict__ slot_of, int n_slots, const uint8_t* __restrict__ host, int H, int I,
    int g, BlockOffsets off, float* __restrict__ hbuf, int32_t* __restrict__ flags) {
  extern __shared__ __align__(16) uint8_t smem[];
  __half* xs = reinterpret_cast<__half*>(smem);
  float* xsum = reinterpret_cast<float*>(smem + (size_t)H * 2);
  float* xback = xsum + H / 32;
  griddep_wait();
  griddep_launch_dependents();
  const int p = blockIdx.y;
  const int t = p / k;
  const int e = ids[p];
  stage_activations(x + (size_t)t * H, H, xs, xsum, xback);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarps + warp;
  if (n >= I) return;
  const uint8_t* blk = expert_block(e, E, slot_of, n_slots, pool, block_bytes, host,
                                    (warp == 0 && lane == 0) ? flags : nullptr);
  if (!blk) {
    if (lane == 0) hbuf[(size_t)p * I + n] = 0.0f;
    return;
  }
  const int nch = H / 32;  // 16-byte chunks per row
  const uint8_t* row = blk + (size_t)n * off.gu_row;
  const uint8_t* qg = row + off.gu_q_gate;
  const uint8_t* qu = row + off.gu_q_up;
  const __half* sz = reinterpret_cast<const __half*>(row + off.gu_sz);  // quads per group

  uint4 wg[NIT], wu[NIT];
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int c = lane + 32 * it;
    if (c < nch) {
      wg[it] = ld_stream_v4(qg + 16 * c);
      wu[it] = ld_stream_v4(qu + 16 * c);
    }
  }
  float ag = 0.0f, au = 0.0f;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int c = lane + 32 * it;
    if (c < nch) {
      const half2* xp = reinterpret_cast<const half2*>(xs + 32 * c);
      const float dg = dot32_scaled(wg[it], xp, xback[c]);
      const float du = dot32_scaled(wu[it], xp, xback[c]);
      const int gi = (32 * c) / g;
      const float xsm = xsum[c];
      ag += __half2float(sz[4 * gi + 0]) * (dg - __half2float(sz[4 * gi + 1]) * xsm);
      au += __half2float(sz[4 * gi + 2]) * (du - __half2float(sz[4 * gi + 3]) * xsm);
    }
  }
  ag = warp_sum(ag);
  au = warp_sum(au);
  if (lane == 0) hbuf[(size_t)p * I + n] = silu_f(ag) * au;
}

// grid (ceil(H / kWarps), T); one warp per output row m, looping over the
// k experts of token t. h of the k pairs is rounded to FP16 (the explicit
// rounding point before the down projection) and staged in shared memory.
__global__ void __launch_bounds__(kWarps * 32) down_gemv_kernel(
    const float* __restrict__ hbuf, const int32_t* __restrict__ ids,
    const float* __restrict__ wts, int k, int E, const uint8_t* __restrict__ pool,
    size_t block_bytes, const int32_t* __restrict__ slot_of, int n_slots,
    const uint8_t* __restrict__ host, int H, int I, int g, BlockOffsets off,
    const __half* __restrict__ y_shared,
    __half* __restrict__ y, int32_t* __restrict__ flags) {
  extern __shared__ __align__(16) uint8_t smem[];
  __half* hs = reinterpret_cast<__half*>(smem);                       // [k][I]
  float* hsum = reinterpret_cast<float*>(smem + (size_t)k * I * 2);   // [k][I/32]
  float* hback = hsum + (size_t)k * (I / 32);                         // [k][I/32]
  const uint8_t** blks = reinterpret_cast<const uint8_t**>(hback + (size_t)k * (I / 32));  // [k]
  float* wj = reinterpret_cast<float*>(blks + k);                     // [k]
  const int t = blockIdx.y;
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x < k) {
    const int p = t * k + threadIdx.x;
    blks[threadIdx.x] = expert_block(ids[p], E, slot_of, n_slots, pool, block_bytes, host,
                                     blockIdx.x == 0 ? flags : nullptr);
    wj[threadIdx.x] = wts[p];
  }
  // h of the k pairs of token t: [k][I] floats, contiguous.
  stage_rounded(hbuf + (size_t)t * k * I, k * I, hs, hsum, hback);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * kWarps + warp;
  if (m >= H) return;
  const int nch = I / 32;         // 16-byte chunks per down row
  const int ntask = k * nch;      // (expert, chunk) tasks of this row
  float acc = 0.0f;
  for (int base = 0; base < ntask; base += 32 * 4) {
    uint4 w[4];
    int jj[4], cc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int task = base + lane + 32 * u;
      jj[u] = -1;
      if (task < ntask) {
        const int j = task / nch, c = task - j * nch;
        const uint8_t* blk = blks[j];
        if (blk) {
          jj[u] = j;
          cc[u] = c;
          w[u] = ld_stream_v4(blk + off.d_offset + (size_t)m * off.d_row + off.d_q + 16 * c);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (jj[u] >= 0) {
        const int j = jj[u], c = cc[u];
        const uint8_t* blk = blks[j];
        const int gi = (32 * c) / g;
        const uint8_t* drow = blk + off.d_offset + (size_t)m * off.d_row;
        const __half* dsz = reinterpret_cast<const __half*>(drow + off.d_sz);
        const float s = __half2float(dsz[2 * gi]);
        const float z = __half2float(dsz[2 * gi + 1]);
        const half2* hp = reinterpret_cast<const half2*>(hs + (size_t)j * I + 32 * c);
        const float d = dot32_scaled(w[u], hp, hback[j * nch + c]);
        acc += wj[j] * (s * (d - z * hsum[j * nch + c]));
      }
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    float v = acc;
    if (y_shared) v += __half2float(y_shared[(size_t)t * H + m]);
    y[(size_t)t * H + m] = __float2half_rn(v);
  }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

size_t gemv_workspace_bytes(int H, int I, int T, int k) {
  (void)H;
  return ws_scratch_offset(T * k) + (size_t)T * k * I * sizeof(float);
}

int gemv_forward(const ForwardArgs& a) {
  const int H = a.H, I = a.I, g = a.g, T = a.T, k = a.k;
  float* hbuf = reinterpret_cast<float*>(static_cast<uint8_t*>(a.ws) + ws_scratch_offset(T * k));
  int32_t* flags = static_cast<int32_t*>(a.ws);
  const size_t smem_a = (size_t)H * 2 + (size_t)(H / 32) * 8;
  const size_t smem_b = (size_t)k * I * 2 + (size_t)k * (I / 32) * 8 + (size_t)k * sizeof(void*) + (size_t)k * 4;
  if (smem_b > 200 * 1024)
    return fail(MOE_ERR_UNSUPPORTED, "GEMV path: k*I = %d too large for one block's shared memory", k * I);
  const dim3 grid_a((I + kWarps - 1) / kWarps, T * k);
  cudaError_t e;
  const int nit = (H / 32 + 31) / 32;
  if (nit <= 1)
    e = launch_pdl(gateup_gemv_kernel<1>, grid_a, dim3(kWarps * 32), smem_a, a.stream,
                   a.x, a.ids, k, a.E, a.pool, a.block_bytes, a.slot_of, a.n_slots, a.host, H, I, g,
                   a.off, hbuf, flags);
  else if (nit <= 2)
    e = launch_pdl(gateup_gemv_kernel<2>, grid_a, dim3(kWarps * 32), smem_a, a.stream,
                   a.x, a.ids, k, a.E, a.pool, a.block_bytes, a.slot_of, a.n_slots, a.host, H, I, g,
                   a.off, hbuf, flags);
  else if (nit <= 4)
    e = launch_pdl(gateup_gemv_kernel<4>, grid_a, dim3(kWarps * 32), smem_a, a.stream,
                   a.x, a.ids, k, a.E, a.pool, a.block_bytes, a.slot_of, a.n_slots, a.host, H, I, g,
                   a.off, hbuf, flags);
  else
    e = launch_pdl(gateup_gemv_kernel<8>, grid_a, dim3(kWarps * 32), smem_a, a.stream,
                   a.x, a.ids, k, a.E, a.pool, a.block_bytes, a.slot_of, a.n_slots, a.host, H, I, g,
                   a.off, hbuf, flags);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "gateup_gemv launch: %s", cudaGetErrorString(e));

  if (smem_b > 48 * 1024) {
    e = cudaFuncSetAttribute(down_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_b);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "down_gemv smem attr: %s", cudaGetErrorString(e));
  }
  const dim3 grid_b((H + kWarps - 1) / kWarps, T);
  e = launch_pdl(down_gemv_kernel, grid_b, dim3(kWarps * 32), smem_b, a.stream, (const float*)hbuf,
                 a.ids, a.weights, k, a.E, a.pool, a.block_bytes, a.slot_of, a.n_slots, a.host, H, I, g,
                 a.off, a.y_shared, a.y, flags);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "down_gemv launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace moe
