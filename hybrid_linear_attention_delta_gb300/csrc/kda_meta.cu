// kda_meta.cu -- per-call prefill plan, built on the device in one launch.
//
// The Day-0 integration page ("Kimi K3 + vLLM: Inside the Day-0 Production
// Integration", section "Separate Prefill/Decode Code Paths") reports that
// preparing KDA metadata with chains of small eager host-driven ops cost
// 870 us per step at batch 1 and 34 us once fused.  Here the whole plan is one
// single-CTA kernel that reads cu_seqlens and init_slots where they already
// live (device memory) and writes the plan into the workspace:
//   * validates cu_seqlens (starts at 0, non-decreasing, ends at T_total);
//   * validates {src, dst} slots, claims every dst for this call, and rejects
//     duplicate destinations and sources that another sequence overwrites;
//   * computes each sequence's first snapshot index (exclusive scan of
//     floor(L_b / snap_interval)) and checks it against the snaps buffer;
//   * with a retention map, range checks and claims the pool slot of every
//     retained snapshot (one thread per snapshot), so that a snapshot slot
//     shared with another snapshot, a destination or a source is refused;
//   * orders sequences longest first, so the longest serial chains start
//     first on a skewed varlen batch.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kMetaThreads = 256;
constexpr int kMaxSortedB = 8192;  // longest-first ordering up to this batch size

__global__ void __launch_bounds__(kMetaThreads) meta_kernel(PrefillPlan p) {
  const int tid = threadIdx.x;
  const int B = p.B;
  __shared__ long long carry;

  // 1. cu_seqlens
  int bad = 0;
  for (int b = tid; b < B; b += kMetaThreads)
    if (p.cu_seqlens[b + 1] < p.cu_seqlens[b]) bad = 1;
  if (tid == 0 && (p.cu_seqlens[0] != 0 || p.cu_seqlens[B] != p.T_total)) bad = 1;
  bad = __syncthreads_or(bad);
  if (bad) {
    if (tid == 0) raise_error(p.err, ERR_BAD_CU);
    if (tid == 0 && p.coop_hdr) p.coop_hdr[0] = p.coop_hdr[1] = p.coop_hdr[2] = 0;
    for (int b = tid; b < B; b += kMetaThreads) {
      SeqMeta m = {0, 0, -1, 0, 0, 0, 0};
      p.meta[b] = m;
      p.order[b] = b;
    }
    return;
  }

  // 2. slots: range, then claim destinations
  const int64_t claim_stride = (int64_t)p.H * kClaimsPerState;
  for (int b = tid; b < B; b += kMetaThreads) {
    const int src = p.init_slots[2 * b], dst = p.init_slots[2 * b + 1];
    int ok = (src >= -1 && src < p.n_slots && dst >= 0 && dst < p.n_slots);
    if (!ok) raise_error(p.err, ERR_BAD_SLOT);
    if (ok && !claim_state(p.claims, (int64_t)dst * claim_stride, p.epoch)) {
      raise_error(p.err, ERR_DUP_SLOT);
      ok = 0;
    }
    SeqMeta m;
    m.tok0 = p.cu_seqlens[b];
    m.len = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
    m.src = src;
    m.dst = dst;
    m.snap_off = 0;
    m.ok = ok;
    m.pad = 0;
    p.meta[b] = m;
  }
  __threadfence_block();
  __syncthreads();

  // 3. snapshot offsets: exclusive scan of floor(len / interval), tile by tile
  if (tid == 0) carry = 0;
  __syncthreads();
  __shared__ long long scan[kMetaThreads];
  for (int base = 0; base < B; base += kMetaThreads) {
    const int b = base + tid;
    long long cnt = 0;
    if (b < B && p.snap_interval > 0) cnt = p.meta[b].len / p.snap_interval;
    scan[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < kMetaThreads; off <<= 1) {
      const long long add = tid >= off ? scan[tid - off] : 0;
      __syncthreads();
      scan[tid] += add;
      __syncthreads();
    }
    if (b < B) {
      const long long first = carry + scan[tid] - cnt;
      p.meta[b].snap_off = first;
      if (cnt > 0 && first + cnt > p.snaps_capacity) {
        raise_error(p.err, ERR_SNAP_CAPACITY);
        p.meta[b].ok = 0;
      }
    }
    __syncthreads();
    if (tid == kMetaThreads - 1) carry += scan[tid];
    __syncthreads();
  }

  // 4. retention map: snapshot s belongs to the last sequence whose first
  // snapshot index is <= s (that sequence has at least one snapshot); a slot
  // out of range or already claimed in this call refuses the sequence
  if (p.snap_slots) {
    const long long n_snap = carry < p.snaps_capacity ? carry : p.snaps_capacity;
    for (long long s = tid; s < n_snap; s += kMetaThreads) {
      const int slot = p.snap_slots[s];
      if (slot == -1) continue;
      int lo = 0, hi = B - 1;
      while (lo < hi) {  // largest b with snap_off[b] <= s
        const int mid = (lo + hi + 1) >> 1;
        if (p.meta[mid].snap_off <= s) lo = mid; else hi = mid - 1;
      }
      if (slot < -1 || slot >= p.n_slots) {
        raise_error(p.err, ERR_BAD_SLOT);
        p.meta[lo].ok = 0;
      } else if (!claim_state(p.claims, (int64_t)slot * claim_stride, p.epoch)) {
        raise_error(p.err, ERR_DUP_SLOT);
        p.meta[lo].ok = 0;
      }
    }
    __threadfence_block();
    __syncthreads();
  }

  // 5. a source that another sequence of this call overwrites (as its
  // destination or a retained snapshot) would race
  for (int b = tid; b < B; b += kMetaThreads) {
    SeqMeta m = p.meta[b];
    if (m.ok && m.src >= 0 && m.src != m.dst) {
      const uint32_t stamp = atomicAdd(p.claims + (int64_t)m.src * claim_stride, 0u);
      if (stamp == p.epoch) {
        raise_error(p.err, ERR_DUP_SLOT);
        p.meta[b].ok = 0;
      }
    }
  }
  __syncthreads();

  // 6. cooperative-mode header: ticket and abort cleared, longest sequence in
  // chunks; ready / consumed flags cleared (the workspace may have held other
  // data at their place in a call with other sizes)
  if (p.coop_hdr) {
    const int nflags = 3 * p.B * p.H * kCoopRing;  // ready, consumed x 2
    for (int i = tid; i < nflags; i += kMetaThreads) p.coop_flags[i] = 0ull;
    int mx = 0;
    for (int b = tid; b < B; b += kMetaThreads) {
      const SeqMeta m = p.meta[b];
      if (m.ok) mx = max(mx, (m.len + 63) / 64);
    }
    for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    __shared__ int wmax[kMetaThreads / 32];
    if ((tid & 31) == 0) wmax[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kMetaThreads / 32; ++w) mx = max(mx, wmax[w]);
      p.coop_hdr[0] = 0;
      p.coop_hdr[1] = 0;
      p.coop_hdr[2] = (uint32_t)mx;
    }
  }

  // 7. longest first (stable: ties keep batch order)
  for (int b = tid; b < B; b += kMetaThreads) {
    int rank = b;
    if (B <= kMaxSortedB) {
      const int lb = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
      rank = 0;
      for (int c = 0; c < B; ++c) {
        const int lc = p.cu_seqlens[c + 1] - p.cu_seqlens[c];
        rank += (lc > lb) || (lc == lb && c < b);
      }
    }
    p.order[rank] = b;
  }
}

}  // namespace

cudaError_t launch_meta(const PrefillPlan &p) {
  meta_kernel<<<1, kMetaThreads, 0, p.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
