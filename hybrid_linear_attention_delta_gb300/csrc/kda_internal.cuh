// kda_internal.cuh -- shared definitions of the libkda.so CUDA sources.
//
// Workspace layout (caller-owned device memory, zero-filled once after
// allocation, see include/kda.h):
//   [0, 256)                 header: uint32 error bits (sticky)
//   [256, +align(B*32))      SeqMeta[B]   per-sequence plan written by the metadata kernel
//   [.., +align(B*4))        int32 order[B]: sequences, longest first
//   [.., +align(n_slots*H*4*4)) uint32 claims: epoch stamps that detect two
//                            sequences of one call writing the same state
//   [.., +align(B*H*4))      uint32 rerun[B*H] (prefill, indexed by longest-first
//                            rank * H + head): the call's epoch when the chunked
//                            kernel found a decay beyond its exponent range in
//                            that (sequence, head); the exact token-recurrent
//                            kernel then recomputes the unit in the same call
//   when B*H <= kCoopMaxUnits, the cooperative prefill's section:
//   [.., +256)               uint32 ticket, abort word, longest sequence in chunks
//   [.., +align(B*H*R*24))   u64 ready[B*H][R] and consumed[2][B*H][R] flags (R =
//                            kCoopRing; one consumed flag per chain CTA of a pair)
//   [.., +B*H*R*74752)       package ring, R chunk packages per (sequence, head)
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

enum ErrBits : uint32_t {
  ERR_BAD_SLOT = 1u,
  ERR_DUP_SLOT = 2u,
  ERR_BAD_CU = 4u,
  ERR_SNAP_CAPACITY = 8u,
  ERR_TIMEOUT = 16u,
  ERR_RESERVED_32 = 32u,  // no longer raised: such units are recomputed exactly
  ERR_BAD_ACCEPT = 64u,
};

struct SeqMeta {
  int32_t tok0;      // first packed token row
  int32_t len;       // tokens in this segment
  int32_t src;       // initial state slot, -1 = zero
  int32_t dst;       // final state slot
  int64_t snap_off;  // index of this sequence's first snapshot
  int32_t ok;        // 0: skip every write of this sequence (a device check failed)
  int32_t pad;
};
static_assert(sizeof(SeqMeta) == 32, "SeqMeta is 32 bytes");

constexpr int kClaimsPerState = 4;  // one claim word per (slot, head, column block)

// Cooperative prefill (few (sequence, head) pairs): per pair a ring of chunk
// packages handed from producer CTAs to the pair's state-carrying CTA.
constexpr int kCoopMaxUnits = 64;      // (sequence, head) pairs it serves at most
// packages in flight per pair.  With the half chains' outputs leaving through TMA
// stores, 12 measured 4% faster than 6 on the 2^20-token prefill (20.71 -> 19.85 ms
// back to back on one GPU; 9 and 24 within 0.1% of 12) and the same on the 8k-token
// one.  (With one loader per chain CTA, 6 had been 1% faster than 8 and 8% faster
// than 16 on the 8k-token prefill: a deeper ring lets the producers run ahead of
// all pairs together, and its packages go cold in L2.)
constexpr int kCoopRing = 12;
constexpr size_t kCoopPkgBytes = 74752;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WorkspaceLayout {
  size_t meta_off, order_off, claims_off, rerun_off, coop_off, coop_flags_off, coop_ring_off,
      total;
  int64_t coop_units;
  __host__ __device__ WorkspaceLayout(int64_t B, int64_t H, int64_t n_slots) {
    meta_off = 256;
    order_off = meta_off + align256((size_t)B * sizeof(SeqMeta));
    claims_off = order_off + align256((size_t)B * sizeof(int32_t));
    rerun_off = claims_off + align256((size_t)n_slots * H * kClaimsPerState * sizeof(uint32_t));
    coop_off = rerun_off + align256((size_t)B * H * sizeof(uint32_t));
    coop_units = (B * H <= kCoopMaxUnits) ? B * H : 0;
    // header (ticket, abort, max chunks) | ready[u][ring] | consumed[u][ring] | ring
    coop_flags_off = coop_off + 256;
    coop_ring_off = coop_flags_off + align256((size_t)coop_units * kCoopRing * 24);
    total = coop_units ? coop_ring_off + (size_t)coop_units * kCoopRing * kCoopPkgBytes
                       : coop_off;
  }
};

// ---------------------------------------------------------------- element io
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void raise_error(uint32_t *err, uint32_t bits) {
  atomicOr(err, bits);
}

// Claims (slot, head, block) for this call; returns false when another CTA of
// the same call already claimed it (two sequences would write one state).
__device__ __forceinline__ bool claim_state(uint32_t *claims, int64_t index, uint32_t epoch) {
  return atomicExch(claims + index, epoch) != epoch;
}

// Where snapshot s of head h is written: the dense snapshot buffer, or, when
// the caller passed a retention map (snap_slots), the pool slot snap_slots[s]
// (nullptr: this snapshot is not retained).  Slots in the map were range
// checked and claimed by the plan kernel; a sequence with a bad one is
// skipped before any kernel gets here.
__device__ __forceinline__ float *snapshot_base(float *snaps, const int32_t *snap_slots,
                                                float *pool, int64_t s, int H, int h,
                                                int64_t state_elems) {
  if (snap_slots) {
    const int slot = snap_slots[s];
    return slot >= 0 ? pool + ((int64_t)slot * H + h) * state_elems : nullptr;
  }
  return snaps + (s * H + h) * state_elems;
}

// ---------------------------------------------------------------- launchers
struct PrefillPlan {
  const void *q, *k, *v, *g, *beta;
  const int32_t *cu_seqlens, *init_slots;
  float *pool;
  void *out;
  float *snaps;
  // retention map [snaps_capacity] (kda_prefill_varlen_retain): snapshot s
  // goes to pool slot snap_slots[s], or nowhere when it is -1; NULL: the
  // dense snaps buffer
  const int32_t *snap_slots;
  int32_t snap_interval;
  int64_t snaps_capacity;
  int32_t B, T_total, H, dk, dv, n_slots, dtype;
  uint32_t *err;
  SeqMeta *meta;
  int32_t *order;
  uint32_t *claims;
  // [B*H] per (longest-first rank, head): == epoch when the chunked kernel
  // handed the unit to the exact recurrent kernel (decay beyond its range)
  uint32_t *rerun;
  uint32_t epoch;
  cudaStream_t stream;
  // cooperative mode (null when the workspace has no room for it)
  uint32_t *coop_hdr;           // [0] ticket, [1] abort, [2] max chunks per sequence
  unsigned long long *coop_flags;  // ready[units][ring] then consumed[units][ring]
  uint8_t *coop_ring;           // [units][ring][kCoopPkgBytes]
};

struct DecodePlan {
  const void *q, *k, *v, *g, *beta;
  const int32_t *slot_ids;
  float *pool;
  void *out;
  float *per_tok;
  int32_t N, n_tok, H, dk, dv, n_slots, dtype;
  uint32_t *err;
  uint32_t *claims;
  uint32_t epoch;
  cudaStream_t stream;
  // speculative verify with commit (spec != 0): sequence n first replays the
  // accepted[n] leading tokens of the previous verify step (rows n * n_prev +
  // j of k_prev, v_prev, g_prev, beta_prev), writes the slot once after them,
  // then runs this step's n_tok tokens for their outputs only (the slot is not
  // advanced past the committed state).  accepted may be NULL when n_prev == 0.
  int32_t spec, n_prev;
  const void *k_prev, *v_prev, *g_prev, *beta_prev;
  const int32_t *accepted;
};

// The layer around the recurrence (kda_prefill_varlen_fused / kda_decode_fused):
// the short causal convolution of the raw q, k, v channels with its state in
// a slot-indexed pool, and the gated RMSNorm of the outputs.
struct FusedParams {
  const void *xq, *xk, *xv;  // raw inputs [T][H][dk], [T][H][dk], [T][H][dv]
  const void *gate;          // [T][H][dv] output gate logits
  const float *conv_w;       // [H][2 dk + dv][kConvW] taps, channel order q | k | v
  const float *norm_w;       // [dv]
  void *conv_pool;           // [n_slots][H][2 dk + dv][kConvW - 1], oldest first
  int32_t act;               // 0: none, 1: SiLU
  float eps;
};
constexpr int kConvW = 4;

cudaError_t launch_meta(const PrefillPlan &p);
// prefill side, in stream order: the convolution of p's batch into q, k, v
// (p.q, p.k, p.v point at the caller's scratch), then the new convolution
// states (after it, so that src == dst is safe), and, after the prefill, the
// gated RMSNorm of o (scratch) into out
cudaError_t launch_conv_prefill(const PrefillPlan &p, const FusedParams &f);
cudaError_t launch_conv_state(const PrefillPlan &p, const FusedParams &f);
cudaError_t launch_rms_gate(const PrefillPlan &p, const FusedParams &f, const void *o, void *out);
// decode: one launch per call, dk = dv = 128 (p.q/k/v unused: f.xq/xk/xv)
cudaError_t launch_decode_fused(const DecodePlan &p, const FusedParams &f);
// rerun_only: recompute only the units that the chunked kernel flagged in
// p.rerun with the call's epoch (every other CTA returns at once)
cudaError_t launch_recurrent_prefill(const PrefillPlan &p, bool rerun_only = false);
cudaError_t launch_recurrent_decode(const DecodePlan &p);
cudaError_t launch_decode128(const DecodePlan &p);
// The chunked tensor-core prefill: whether it applies to these shapes, whether
// its cooperative mode can run, and the launch (mode: which variant).
enum ChunkMode { kChunkAuto = 0, kChunkPerState = 1, kChunkCoop = 2, kChunkCoopHalves = 3 };
bool chunked_supported(const PrefillPlan &p);
// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) once per
// (function, device) in this process (thread-safe)
cudaError_t set_smem_limit_once(const void *func, int bytes);
bool coop_supported(const PrefillPlan &p);
// the cooperative mode with two chain CTAs per (sequence, head), one per half
// of the value columns
bool coop_halves_supported(const PrefillPlan &p);
cudaError_t launch_chunked_prefill(const PrefillPlan &p, int mode);

}  // namespace kda
