// kda_decode.cu -- in-place KDA decode for dk = dv = 128 on a slot-indexed
// fp32 state pool (single token, or n_tok tokens of a speculative verify pass
// with the state after each token kept for rollback).
//
// Decode is the fused per-token step of "Kimi K3 on vLLM: Up to 370
// Tokens/sec", section "Kimi Delta Attention: a hybrid recurrent +
// full-attention stack" (a fused CUDA kernel for decode; the multi-token path
// for speculative decoding).  Per token, with S' = Diag(exp g) S:
//     x = S'^T k ,  y = S'^T q            (both reductions in one pass over S')
//     u = beta (v - x) ;  o = S^T q = y + u (k . q) ;  S = S' + k u^T
//
// The step is bound by HBM: one 64 KiB fp32 state is read and written per
// (sequence, head) against ~1 KiB of token data.  One CTA of 256 threads owns
// one state.  Warp w holds rows [16w, 16w+16) and lane l holds columns
// [4l, 4l+4) of those rows, so each row is one 512-byte coalesced 128-bit
// load per warp and the whole state is in flight after 16 loads per thread.
// Reductions over rows are thread-local over 16 rows and then one pass over
// the 8 warps in shared memory; the update and the write-back are in
// registers.  Every state is read exactly once and written once (plus once
// per token when per-token states are requested).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kRowsPerWarp = kD / (kThreads / 32);  // 16

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 2) decode128_kernel(DecodePlan p) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31;
  const int H = p.H;
  const int n = blockIdx.x / H, h = blockIdx.x % H;

  __shared__ int s_slot;
  // su is read as float4: every staging array is 16-byte aligned
  __shared__ __align__(16) float sa[kD];
  __shared__ __align__(16) float sk[kD];
  __shared__ __align__(16) float sq[kD];
  __shared__ __align__(16) float sv[kD];
  __shared__ __align__(16) float su[kD];
  __shared__ __align__(16) float sy[kD];
  __shared__ __align__(16) float redx[kThreads / 32][kD];
  __shared__ __align__(16) float redy[kThreads / 32][kD];
  __shared__ float skq[4], sbeta;

  if (tid == 0) {
    int slot = p.slot_ids[n];
    if (slot < 0 || slot >= p.n_slots) {
      raise_error(p.err, ERR_BAD_SLOT);
      slot = -1;
    } else if (!claim_state(p.claims, ((int64_t)slot * H + h) * kClaimsPerState, p.epoch)) {
      raise_error(p.err, ERR_DUP_SLOT);
      slot = -1;
    }
    s_slot = slot;
  }
  __syncthreads();
  const int slot = s_slot;
  if (slot < 0) return;

  const int64_t kStateElems = (int64_t)kD * kD;
  float *state = p.pool + ((int64_t)slot * H + h) * kStateElems;
  float4 s[kRowsPerWarp];
#pragma unroll
  for (int m = 0; m < kRowsPerWarp; ++m)
    s[m] = __ldcs(reinterpret_cast<const float4 *>(state + (w * kRowsPerWarp + m) * kD) + l);

  const Tin *q = (const Tin *)p.q, *k = (const Tin *)p.k, *g = (const Tin *)p.g;
  const Tin *v = (const Tin *)p.v, *beta = (const Tin *)p.beta;
  Tin *out = (Tin *)p.out;

  for (int j = 0; j < p.n_tok; ++j) {
    const int64_t row = ((int64_t)n * p.n_tok + j) * H + h;
    if (tid < kD) {
      const float kk = to_f32(k[row * kD + tid]);
      const float qq = to_f32(q[row * kD + tid]);
      sk[tid] = kk;
      sq[tid] = qq;
      sa[tid] = expf(to_f32(g[row * kD + tid]));
      float kq = kk * qq;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
      if (l == 0) skq[w] = kq;
    } else {
      sv[tid - kD] = to_f32(v[row * kD + tid - kD]);
      if (tid == kD) sbeta = to_f32(beta[row]);
    }
    __syncthreads();

    // S' = Diag(a) S ; partial x = S'^T k and y = S'^T q over this warp's rows
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
      const int i = w * kRowsPerWarp + m;
      const float ai = sa[i], ki = sk[i], qi = sq[i];
      s[m].x *= ai; s[m].y *= ai; s[m].z *= ai; s[m].w *= ai;
      x.x = fmaf(ki, s[m].x, x.x); x.y = fmaf(ki, s[m].y, x.y);
      x.z = fmaf(ki, s[m].z, x.z); x.w = fmaf(ki, s[m].w, x.w);
      y.x = fmaf(qi, s[m].x, y.x); y.y = fmaf(qi, s[m].y, y.y);
      y.z = fmaf(qi, s[m].z, y.z); y.w = fmaf(qi, s[m].w, y.w);
    }
    *reinterpret_cast<float4 *>(&redx[w][4 * l]) = x;
    *reinterpret_cast<float4 *>(&redy[w][4 * l]) = y;
    __syncthreads();

    if (tid < kD) {
      float xs = 0.f;
#pragma unroll
      for (int ww = 0; ww < kThreads / 32; ++ww) xs += redx[ww][tid];
      su[tid] = sbeta * (sv[tid] - xs);
    } else {
      float ys = 0.f;
#pragma unroll
      for (int ww = 0; ww < kThreads / 32; ++ww) ys += redy[ww][tid - kD];
      sy[tid - kD] = ys;
    }
    __syncthreads();

    if (tid < kD) {
      const float kq = (skq[0] + skq[1]) + (skq[2] + skq[3]);
      out[row * kD + tid] = from_f32<Tin>(fmaf(su[tid], kq, sy[tid]));
    }
    const float4 u4 = *reinterpret_cast<const float4 *>(&su[4 * l]);
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
      const float ki = sk[w * kRowsPerWarp + m];
      s[m].x = fmaf(ki, u4.x, s[m].x); s[m].y = fmaf(ki, u4.y, s[m].y);
      s[m].z = fmaf(ki, u4.z, s[m].z); s[m].w = fmaf(ki, u4.w, s[m].w);
    }
    if (p.per_tok) {
      float *pt = p.per_tok + (((int64_t)n * p.n_tok + j) * H + h) * kStateElems;
#pragma unroll
      for (int m = 0; m < kRowsPerWarp; ++m)
        __stcs(reinterpret_cast<float4 *>(pt + (w * kRowsPerWarp + m) * kD) + l, s[m]);
    }
    __syncthreads();  // the next token's staging overwrites sk, su, sy
  }

#pragma unroll
  for (int m = 0; m < kRowsPerWarp; ++m)
    __stcs(reinterpret_cast<float4 *>(state + (w * kRowsPerWarp + m) * kD) + l, s[m]);
}

}  // namespace

cudaError_t launch_decode128(const DecodePlan &p) {
  if (p.N == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((int64_t)p.N * p.H);
  if (p.dtype == KDA_BF16)
    decode128_kernel<__nv_bfloat16><<<grid, kThreads, 0, p.stream>>>(p);
  else
    decode128_kernel<float><<<grid, kThreads, 0, p.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
