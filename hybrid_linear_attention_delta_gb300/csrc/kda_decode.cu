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
//
// Two kernels share that layout.  A single-token call (the batched decode
// step) stages its one token while the state loads are in flight and ends as
// soon as the state is written: at two CTAs per SM, every cycle between the
// state's arrival and its write-back costs bandwidth.  Multi-token and
// speculative calls stage their tokens' inputs in shared memory 16 at a time,
// all of a tile's loads in flight together, so the serial token steps (two
// barriers each) wait on no global load.
//
// The speculative variant (kda_decode_spec) folds the commit of the previous
// verify step into this one: it replays that step's accepted tokens from
// their k, v, g, beta, writes the state once, and then evaluates this step's
// draft tokens for their outputs only, so a verify step moves one state read
// and one state write instead of a state per draft token.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kRowsPerWarp = kD / (kThreads / 32);  // 16
constexpr int kTileTok = 16;  // tokens staged in shared memory at a time

// a 16-byte vector of token data as fp32
template <typename T> __device__ __forceinline__ void unpack_vec(uint4 r, float *f);
template <> __device__ __forceinline__ void unpack_vec<float>(uint4 r, float *f) {
  f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
  f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
template <> __device__ __forceinline__ void unpack_vec<__nv_bfloat16>(uint4 r, float *f) {
  const uint32_t u[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(u[j] << 16);
    f[2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
  }
}

// One token per (sequence, head) (the batched decode step): the token's
// inputs are staged by the two thread halves while the state loads are in
// flight, and the CTA ends as soon as the state is written back.
template <typename Tin>
__global__ void __launch_bounds__(kThreads, 2) decode128_single_kernel(DecodePlan p) {
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

template <typename Tin, bool SPEC>
__global__ void __launch_bounds__(kThreads, 2) decode128_kernel(DecodePlan p) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31;
  const int H = p.H;
  const int n = blockIdx.x / H, h = blockIdx.x % H;

  __shared__ int s_slot, s_acc;
  // a tile of up to kTileTok tokens staged as fp32 (exp(g) already taken);
  // every array is 16-byte aligned (su is read as float4)
  __shared__ __align__(16) float tk[kTileTok][kD];
  __shared__ __align__(16) float tq[kTileTok][kD];
  __shared__ __align__(16) float ta[kTileTok][kD];
  __shared__ __align__(16) float tv[kTileTok][kD];
  __shared__ float tb[kTileTok];
  __shared__ float kqp[2][kThreads / 32];  // k . q: one partial per warp, two tokens in turn
  __shared__ __align__(16) float su[kD];
  __shared__ __align__(16) float sy[kD];
  __shared__ __align__(16) float redx[kThreads / 32][kD];
  __shared__ __align__(16) float redy[kThreads / 32][kD];

  if (tid == 0) {
    int slot = p.slot_ids[n];
    if (slot < 0 || slot >= p.n_slots) {
      raise_error(p.err, ERR_BAD_SLOT);
      slot = -1;
    } else if (!claim_state(p.claims, ((int64_t)slot * H + h) * kClaimsPerState, p.epoch)) {
      raise_error(p.err, ERR_DUP_SLOT);
      slot = -1;
    }
    int acc = 0;
    if (SPEC && slot >= 0 && p.n_prev > 0) {
      acc = p.accepted[n];
      if (acc < 0 || acc > p.n_prev) {  // the sequence is skipped: nothing written
        raise_error(p.err, ERR_BAD_ACCEPT);
        slot = -1;
      }
    }
    s_slot = slot;
    s_acc = acc;
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

  // The token list of this (sequence, head): first the acc replayed tokens of
  // the previous verify step (speculative form; no q, no output), then this
  // call's n_tok tokens.
  const int acc = SPEC ? s_acc : 0;
  const int total = acc + p.n_tok;
  constexpr int kVecElems = 16 / (int)sizeof(Tin);             // elements per 16-byte vector
  constexpr int kVecs = kD / kVecElems;                         // vectors per 128-element row
  constexpr int kVecPerThread = kTileTok * 4 * kVecs / kThreads;  // 4 (bf16) or 8 (fp32)
  const Tin *q = (const Tin *)p.q, *k = (const Tin *)p.k, *g = (const Tin *)p.g;
  const Tin *v = (const Tin *)p.v, *beta = (const Tin *)p.beta;
  const Tin *kp = (const Tin *)p.k_prev, *gp = (const Tin *)p.g_prev;
  const Tin *vp = (const Tin *)p.v_prev, *bp = (const Tin *)p.beta_prev;
  Tin *out = (Tin *)p.out;
  auto row_of = [&](int t) -> int64_t {  // (token row) * H + h of list entry t
    return SPEC && t < acc ? ((int64_t)n * p.n_prev + t) * H + h
                           : ((int64_t)n * p.n_tok + (t - acc)) * H + h;
  };

  for (int base = 0; base < total; base += kTileTok) {
    const int nt = min(kTileTok, total - base);
    // stage the tile: 16-byte vectors of k, q, g, v (vector j of a row at
    // item ((tt * 4 + array) * kVecs + j)), all loaded into registers before
    // any is converted, so every load of the tile is in flight at once
    {
      uint4 raw[kVecPerThread];
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        const int e = tid + j * kThreads;
        raw[j] = make_uint4(0, 0, 0, 0);
        if (e < nt * 4 * kVecs) {
          const int tt = e / (4 * kVecs), arr = (e / kVecs) % 4, c = e % kVecs, t = base + tt;
          const bool rep = SPEC && t < acc;
          const Tin *src = arr == 0 ? (rep ? kp : k)
                         : arr == 1 ? (rep ? nullptr : q)
                         : arr == 2 ? (rep ? gp : g) : (rep ? vp : v);
          if (src) raw[j] = *reinterpret_cast<const uint4 *>(src + row_of(t) * kD + c * kVecElems);
        }
      }
      if (tid < nt) {
        const int t = base + tid;
        tb[tid] = to_f32(SPEC && t < acc ? bp[row_of(t)] : beta[row_of(t)]);
      }
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        const int e = tid + j * kThreads;
        if (e < nt * 4 * kVecs) {
          const int tt = e / (4 * kVecs), arr = (e / kVecs) % 4, c = e % kVecs;
          float f[kVecElems];
          unpack_vec<Tin>(raw[j], f);
          float *dst = (arr == 0 ? tk[tt] : arr == 1 ? tq[tt] : arr == 2 ? ta[tt] : tv[tt]) +
                       c * kVecElems;
          if (arr == 2) {
#pragma unroll
            for (int x = 0; x < kVecElems; ++x) f[x] = expf(f[x]);
          }
#pragma unroll
          for (int x = 0; x < kVecElems; x += 4)
            *reinterpret_cast<float4 *>(dst + x) = make_float4(f[x], f[x + 1], f[x + 2], f[x + 3]);
        }
      }
    }
    __syncthreads();

    for (int tt = 0; tt < nt; ++tt) {
      const int t = base + tt;
      // S' = Diag(a) S ; partial x = S'^T k and y = S'^T q over this warp's rows
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
      float kq = 0.f;  // k . q over this warp's rows (the same on every lane)
      if (SPEC && t < acc) {  // a replayed token has no query: x only
#pragma unroll
        for (int m = 0; m < kRowsPerWarp; ++m) {
          const int i = w * kRowsPerWarp + m;
          const float ai = ta[tt][i], ki = tk[tt][i];
          s[m].x *= ai; s[m].y *= ai; s[m].z *= ai; s[m].w *= ai;
          x.x = fmaf(ki, s[m].x, x.x); x.y = fmaf(ki, s[m].y, x.y);
          x.z = fmaf(ki, s[m].z, x.z); x.w = fmaf(ki, s[m].w, x.w);
        }
      } else {
#pragma unroll
        for (int m = 0; m < kRowsPerWarp; ++m) {
          const int i = w * kRowsPerWarp + m;
          const float ai = ta[tt][i], ki = tk[tt][i], qi = tq[tt][i];
          kq = fmaf(ki, qi, kq);
          s[m].x *= ai; s[m].y *= ai; s[m].z *= ai; s[m].w *= ai;
          x.x = fmaf(ki, s[m].x, x.x); x.y = fmaf(ki, s[m].y, x.y);
          x.z = fmaf(ki, s[m].z, x.z); x.w = fmaf(ki, s[m].w, x.w);
          y.x = fmaf(qi, s[m].x, y.x); y.y = fmaf(qi, s[m].y, y.y);
          y.z = fmaf(qi, s[m].z, y.z); y.w = fmaf(qi, s[m].w, y.w);
        }
      }
      *reinterpret_cast<float4 *>(&redx[w][4 * l]) = x;
      *reinterpret_cast<float4 *>(&redy[w][4 * l]) = y;
      if (l == 0) kqp[tt & 1][w] = kq;  // read after the next barrier but one
      __syncthreads();

      // u = beta (v - x) and y = S'^T q, reduced over the 8 warps (the next
      // token's partial sums are written only after the barrier below)
      if (tid < kD) {
        float xs = 0.f;
#pragma unroll
        for (int ww = 0; ww < kThreads / 32; ++ww) xs += redx[ww][tid];
        su[tid] = tb[tt] * (tv[tt][tid] - xs);
      } else {
        float ys = 0.f;
#pragma unroll
        for (int ww = 0; ww < kThreads / 32; ++ww) ys += redy[ww][tid - kD];
        sy[tid - kD] = ys;
      }
      __syncthreads();

      // o = y + u (k . q) ; S = S' + k u^T (su and sy are rewritten only
      // after the next token's first barrier)
      if (tid < kD && t >= acc) {
        const float *kw = kqp[tt & 1];
        const float kq = ((kw[0] + kw[1]) + (kw[2] + kw[3])) + ((kw[4] + kw[5]) + (kw[6] + kw[7]));
        out[row_of(t) * kD + tid] = from_f32<Tin>(fmaf(su[tid], kq, sy[tid]));
      }
      const float4 u4 = *reinterpret_cast<const float4 *>(&su[4 * l]);
#pragma unroll
      for (int m = 0; m < kRowsPerWarp; ++m) {
        const float ki = tk[tt][w * kRowsPerWarp + m];
        s[m].x = fmaf(ki, u4.x, s[m].x); s[m].y = fmaf(ki, u4.y, s[m].y);
        s[m].z = fmaf(ki, u4.z, s[m].z); s[m].w = fmaf(ki, u4.w, s[m].w);
      }
      if (SPEC && t == acc - 1) {  // the committed state: the slot's one write
#pragma unroll
        for (int m = 0; m < kRowsPerWarp; ++m)
          __stcs(reinterpret_cast<float4 *>(state + (w * kRowsPerWarp + m) * kD) + l, s[m]);
      }
      if (!SPEC && p.per_tok) {
        float *pt = p.per_tok + row_of(t) * kStateElems;
#pragma unroll
        for (int m = 0; m < kRowsPerWarp; ++m)
          __stcs(reinterpret_cast<float4 *>(pt + (w * kRowsPerWarp + m) * kD) + l, s[m]);
      }
    }
    __syncthreads();  // the next tile's staging overwrites this one
  }

  if (!SPEC) {
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m)
      __stcs(reinterpret_cast<float4 *>(state + (w * kRowsPerWarp + m) * kD) + l, s[m]);
  }
}

}  // namespace

cudaError_t launch_decode128(const DecodePlan &p) {
  if (p.N == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((int64_t)p.N * p.H);
  if (!p.spec && p.n_tok == 1) {
    if (p.dtype == KDA_BF16)
      decode128_single_kernel<__nv_bfloat16><<<grid, kThreads, 0, p.stream>>>(p);
    else
      decode128_single_kernel<float><<<grid, kThreads, 0, p.stream>>>(p);
  } else if (p.spec) {
    if (p.dtype == KDA_BF16)
      decode128_kernel<__nv_bfloat16, true><<<grid, kThreads, 0, p.stream>>>(p);
    else
      decode128_kernel<float, true><<<grid, kThreads, 0, p.stream>>>(p);
  } else if (p.dtype == KDA_BF16) {
    decode128_kernel<__nv_bfloat16, false><<<grid, kThreads, 0, p.stream>>>(p);
  } else {
    decode128_kernel<float, false><<<grid, kThreads, 0, p.stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kda
