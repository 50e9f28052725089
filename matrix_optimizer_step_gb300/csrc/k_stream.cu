// Streaming (HBM-bound) kernels of the owner-side step:
//   momentum  -- buf <- mu*buf + g, u <- g + mu*buf (Nesterov), X0 <- u into
//                the Newton-Schulz workspace (operand dtype, plus an fp32
//                copy on the bf16 path), per-chunk sum of u^2
//   norm      -- per-slice 1/(||u||_F + 1e-7) from the chunk partials
//   update    -- W <- W*(1 - lr*wd) - lr*scale*X, bf16 copy of W
//   adamw     -- the element-wise AdamW step
// DMuon docs, "架构设计" §2 (the owner's optimizer step: momentum, weight
// decay, parameter update) and "Pure DMuon 路由" (AdamW routes; fp32
// master/optimizer state with a bf16 parameter).
//
// Every kernel walks a host-built chunk table: one block per chunk of at
// most kChunkElems elements of one slice/vector.  Groups of 8 elements move
// as 16-byte vectors when the slice allows it (n % 8 == 0 and aligned
// pointers); otherwise a scalar path handles the elements one by one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace dmuon {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void load8_f32(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8_f32_rw(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8_f32(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void load8_bf16(const void* p, float (&v)[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void store8_bf16(void* p, const float (&v)[8]) {
  uint4 q;
  q.x = pack_bf16x2(v[0], v[1]);
  q.y = pack_bf16x2(v[2], v[3]);
  q.z = pack_bf16x2(v[4], v[5]);
  q.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = q;
}

__device__ __forceinline__ float load1(const void* p, int64_t i, int is_bf16) {
  if (is_bf16) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store1(void* p, int64_t i, float v, int is_bf16) {
  if (is_bf16)
    reinterpret_cast<uint16_t*>(p)[i] = to_bf16_bits(v);
  else
    reinterpret_cast<float*>(p)[i] = v;
}

// Deterministic block sum (fixed shuffle tree, then fixed warp order).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  }
  return s;
}

// ------------------------------------------------------------ momentum pass
__global__ void __launch_bounds__(kThreads) momentum_kernel(const SliceDesc* __restrict__ slices,
                                                            const Chunk* __restrict__ chunks,
                                                            float mu, int nesterov, int x_fp32,
                                                            float* __restrict__ partials) {
  __shared__ float red[kThreads / 32];
  const Chunk ch = chunks[blockIdx.x];
  const SliceDesc S = slices[ch.slice];
  const int64_t end = ch.start + ch.count;
  x_fp32 = x_fp32 || S.x_f32;
  float ss = 0.f;
  if (S.vec_ok) {
    const bool dense = (S.ld == S.n);
    for (int64_t e = ch.start + 8 * static_cast<int64_t>(threadIdx.x); e < end;
         e += 8 * kThreads) {
      float g[8], buf[8], u[8];
      if (S.grad_bf16)
        load8_bf16(reinterpret_cast<const uint16_t*>(S.grad) + e, g);
      else
        load8_f32(reinterpret_cast<const float*>(S.grad) + e, g);
      load8_f32_rw(S.momentum + e, buf);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        buf[i] = fmaf(mu, buf[i], g[i]);
        u[i] = nesterov ? fmaf(mu, buf[i], g[i]) : buf[i];
        ss = fmaf(u[i], u[i], ss);
      }
      store8_f32(S.momentum + e, buf);
      int64_t xi = e;
      if (!dense) {
        const int64_t row = e / S.n;
        xi = row * S.ld + (e - row * S.n);
      }
      if (x_fp32)
        store8_f32(reinterpret_cast<float*>(S.x0) + xi, u);
      else
        store8_bf16(reinterpret_cast<uint16_t*>(S.x0) + xi, u);
      if (S.x0lo) {
        uint4 q;
        q.x = pack_bf16x2_remainder(u[0], u[1]);
        q.y = pack_bf16x2_remainder(u[2], u[3]);
        q.z = pack_bf16x2_remainder(u[4], u[5]);
        q.w = pack_bf16x2_remainder(u[6], u[7]);
        *reinterpret_cast<uint4*>(S.x0lo + xi) = q;
      }
    }
  } else {
    for (int64_t e = ch.start + threadIdx.x; e < end; e += kThreads) {
      const float g = load1(S.grad, e, S.grad_bf16);
      const float b = fmaf(mu, S.momentum[e], g);
      const float u = nesterov ? fmaf(mu, b, g) : b;
      S.momentum[e] = b;
      ss = fmaf(u, u, ss);
      const int64_t row = e / S.n;
      const int64_t xi = row * S.ld + (e - row * S.n);
      store1(S.x0, xi, u, !x_fp32);
      if (S.x0lo) S.x0lo[xi] = to_bf16_bits(bf16_remainder(u));
    }
  }
  const float tot = block_sum(ss, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = tot;
}

// ---------------------------------------------------------------- norm pass
__global__ void norm_kernel(const SliceDesc* __restrict__ slices, int n_slices,
                            const float* __restrict__ partials, float* __restrict__ inv_norm) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n_slices) return;
  const int cb = slices[w].chunk_begin, ce = slices[w].chunk_end;
  double s = 0.0;
  for (int c = cb + lane; c < ce; c += 32) s += static_cast<double>(partials[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) inv_norm[w] = static_cast<float>(1.0 / (sqrt(s) + 1e-7));
}

// -------------------------------------------------------------- update pass
__global__ void __launch_bounds__(kThreads) update_kernel(const SliceDesc* __restrict__ slices,
                                                          const Chunk* __restrict__ chunks,
                                                          float lr, float wd, int x_fp32,
                                                          const float* __restrict__ xscale) {
  const Chunk ch = chunks[blockIdx.x];
  const SliceDesc S = slices[ch.slice];
  const int64_t end = ch.start + ch.count;
  x_fp32 = x_fp32 || S.x_f32;
  const float decay = 1.0f - lr * wd;
  float step = lr * S.shape_scale;
  if (xscale) step *= xscale[ch.slice];
  if (S.vec_ok) {
    const bool dense = (S.ld == S.n);
    for (int64_t e = ch.start + 8 * static_cast<int64_t>(threadIdx.x); e < end;
         e += 8 * kThreads) {
      int64_t xi = e;
      if (!dense) {
        const int64_t row = e / S.n;
        xi = row * S.ld + (e - row * S.n);
      }
      float x[8], w[8];
      if (x_fp32)
        load8_f32(reinterpret_cast<const float*>(S.xk) + xi, x);
      else
        load8_bf16(reinterpret_cast<const uint16_t*>(S.xk) + xi, x);
      load8_f32_rw(S.master + e, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = fmaf(-step, x[i], w[i] * decay);
      store8_f32(S.master + e, w);
      if (S.param) store8_bf16(S.param + e, w);
    }
  } else {
    for (int64_t e = ch.start + threadIdx.x; e < end; e += kThreads) {
      const int64_t row = e / S.n;
      const float x = load1(S.xk, row * S.ld + (e - row * S.n), !x_fp32);
      const float w = fmaf(-step, x, S.master[e] * decay);
      S.master[e] = w;
      if (S.param) S.param[e] = to_bf16_bits(w);
    }
  }
}

// --------------------------------------------------------------- AdamW pass
__device__ __forceinline__ float adamw_elem(float g, float& w, float& m, float& v, float b1,
                                            float b2, float eps, float decay, float step_size,
                                            float bc2_sqrt) {
  m = fmaf(b1, m, (1.0f - b1) * g);
  v = fmaf(b2, v, (1.0f - b2) * g * g);
  const float denom = sqrtf(v) / bc2_sqrt + eps;
  w = fmaf(-step_size, m / denom, w * decay);
  return w;
}

__global__ void __launch_bounds__(kThreads) adamw_kernel(const VecDesc* __restrict__ vecs,
                                                         const Chunk* __restrict__ chunks,
                                                         float lr, float b1, float b2, float eps,
                                                         float wd, float bc1, float bc2_sqrt) {
  const Chunk ch = chunks[blockIdx.x];
  const VecDesc V = vecs[ch.slice];
  const int64_t end = ch.start + ch.count;
  const float decay = 1.0f - lr * wd;
  const float step_size = lr / bc1;
  int64_t e0 = ch.start;
  if (V.vec_ok) {
    const int64_t vec_end = ch.start + (static_cast<int64_t>(ch.count) & ~int64_t(7));
    for (int64_t e = ch.start + 8 * static_cast<int64_t>(threadIdx.x); e < vec_end;
         e += 8 * kThreads) {
      float g[8], w[8], m[8], v[8];
      if (V.grad_bf16)
        load8_bf16(reinterpret_cast<const uint16_t*>(V.grad) + e, g);
      else
        load8_f32(reinterpret_cast<const float*>(V.grad) + e, g);
      load8_f32_rw(V.master + e, w);
      load8_f32_rw(V.exp_avg + e, m);
      load8_f32_rw(V.exp_avg_sq + e, v);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        adamw_elem(g[i], w[i], m[i], v[i], b1, b2, eps, decay, step_size, bc2_sqrt);
      store8_f32(V.master + e, w);
      store8_f32(V.exp_avg + e, m);
      store8_f32(V.exp_avg_sq + e, v);
      if (V.param) store8_bf16(V.param + e, w);
    }
    e0 = vec_end;
  }
  for (int64_t e = e0 + threadIdx.x; e < end; e += kThreads) {
    float w = V.master[e], m = V.exp_avg[e], v = V.exp_avg_sq[e];
    adamw_elem(load1(V.grad, e, V.grad_bf16), w, m, v, b1, b2, eps, decay, step_size, bc2_sqrt);
    V.master[e] = w;
    V.exp_avg[e] = m;
    V.exp_avg_sq[e] = v;
    if (V.param) V.param[e] = to_bf16_bits(w);
  }
}

// ------------------------------------------------- bounded-wait self test
// Waits on a barrier that nothing completes; the bounded wait must give up,
// record kErrTimeoutSelftest and let the kernel return.
__global__ void selftest_wait_kernel(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, kErrTimeoutSelftest, limit_ns);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_momentum(const SliceDesc* slices, const Chunk* chunks, int n_chunks, float mu,
                            int nesterov, int x_fp32, float* partials, cudaStream_t st) {
  if (n_chunks <= 0) return cudaSuccess;
  momentum_kernel<<<n_chunks, kThreads, 0, st>>>(slices, chunks, mu, nesterov, x_fp32, partials);
  return cudaGetLastError();
}

cudaError_t launch_norm(const SliceDesc* slices, int n_slices, const float* partials,
                        float* inv_norm, cudaStream_t st) {
  if (n_slices <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int blocks = (n_slices + warps_per_block - 1) / warps_per_block;
  norm_kernel<<<blocks, warps_per_block * 32, 0, st>>>(slices, n_slices, partials, inv_norm);
  return cudaGetLastError();
}

cudaError_t launch_update(const SliceDesc* slices, const Chunk* chunks, int n_chunks, float lr,
                          float wd, int x_fp32, const float* xscale, cudaStream_t st) {
  if (n_chunks <= 0) return cudaSuccess;
  update_kernel<<<n_chunks, kThreads, 0, st>>>(slices, chunks, lr, wd, x_fp32, xscale);
  return cudaGetLastError();
}

cudaError_t launch_adamw(const VecDesc* vecs, const Chunk* chunks, int n_chunks, float lr,
                         float beta1, float beta2, float eps, float wd, float bc1, float bc2_sqrt,
                         cudaStream_t st) {
  if (n_chunks <= 0) return cudaSuccess;
  adamw_kernel<<<n_chunks, kThreads, 0, st>>>(vecs, chunks, lr, beta1, beta2, eps, wd, bc1,
                                              bc2_sqrt);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int* err, long long timeout_ns, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(err, static_cast<unsigned long long>(timeout_ns));
  return cudaGetLastError();
}

}  // namespace dmuon
