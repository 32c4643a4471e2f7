// prefetch_rows.cuh -- the copy step of the fused lossless prefetch, shared by the
// decode indexer (candidates from the threshold test of each scored tile) and the
// prefill indexer (candidates from the approximate top-k of each query block).
//
// ECHO review (marsggbo.github.io, "OSDI'26 | ECHO"), section 6.1: a candidate takes
// a ticket from a global counter whose bound is proportional to the context length,
// and its latent-KV row is loaded from the pinned host pool while scoring continues.
// Destinations: the HBM staging area (per-request counters and caps), or, direct to
// slot, the GPU-pool slots the last recall set aside (one counter over the reserve;
// the row's HostTokenToGPU entry is claimed with a compare-and-swap, so a row is
// placed once, and the row is resident from then on).
#pragma once

#include "echo_common.cuh"

namespace echo {

constexpr int kPfRowsPerBatch = 4;  // rows one prefetch warp keeps in flight

__device__ __forceinline__ int clamp_ctx(int32_t L, int L_max) { return L < 0 ? 0 : (L > L_max ? L_max : L); }

// One warp.  Lanes with cand = true hold a candidate: a token of request b whose host
// row h was found not resident.  Tickets, then the rows, kPfRowsPerBatch at a time
// (9 16-byte loads in flight per lane); a row whose ticket is past the bound is read
// but not stored.  res_len is the reserve length (direct to slot); res_full (warp
// uniform) records that this warp has seen the tickets pass it, after which its later
// candidates are dropped unread.  Params needs the fields of the prefetch (host_kv,
// host_to_gpu, stage_*, cap_div, ctx_len, L_max, reserve, reserve_ctl, to_host, prio,
// gpu_kv, n_g, status).
template <class Params>
__device__ __forceinline__ void prefetch_copy_batch(const Params &P, bool cand, int32_t h, int b, int32_t res_len,
                                                    bool &res_full) {
  const int lane = threadIdx.x & 31;
  const bool direct = P.reserve != nullptr;
  const int4 *host = reinterpret_cast<const int4 *>(P.host_kv);
  int4 *dst_rows = reinterpret_cast<int4 *>(direct ? P.gpu_kv : P.stage_rows);
  int32_t dst = -1;
  const uint32_t cmask = __ballot_sync(0xffffffffu, cand);
  if (direct && res_full) {
    if (cmask && lane == 0) set_status(P.status, ECHO_DEV_PREFETCH_CAP_HIT);
    return;
  }
  // tickets: one atomic per request among the candidates (staging) or one for the
  // warp's candidates (direct to slot); the result is needed only for the
  // destinations, so the first host loads below start before it returns
  uint32_t grp = 0;
  int leader = 0, base = 0;
  if (cand) {
    grp = direct ? cmask : __match_any_sync(cmask, b);  // candidates sharing a counter
    leader = __ffs(grp) - 1;
    if (lane == leader) base = atomicAdd(direct ? P.reserve_ctl : P.stage_count + b, __popc(grp));
  }
  // ---- copy the candidate rows, kPfRowsPerBatch at a time (9 16-byte loads in flight
  // per lane); a row whose ticket is past the cap is read but not stored
  uint32_t rem = cmask;
  bool have_tickets = false;
  while (rem) {
    int32_t hr[kPfRowsPerBatch], sl[kPfRowsPerBatch], dr[kPfRowsPerBatch];
    int cnt = 0;
#pragma unroll
    for (int r = 0; r < kPfRowsPerBatch; ++r) {
      int src_lane = 0;
      if (rem) {
        src_lane = __ffs(rem) - 1;
        rem &= rem - 1;
        ++cnt;
      }
      sl[r] = src_lane;
      hr[r] = __shfl_sync(0xffffffffu, h, src_lane);
    }
    constexpr int kPer = (kPfRowsPerBatch * kKvChunks + 31) / 32;
    int4 buf[kPer];
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int idx = m * 32 + lane;
      const int r = idx / kKvChunks, c = idx % kKvChunks;
      if (r < cnt) buf[m] = __ldcs(host + static_cast<size_t>(pick_reg(hr, r)) * kKvChunks + c);
    }
    if (!have_tickets) {
      have_tickets = true;
      if (direct) {
        // ticket t places the row in reserved slot reserve[t]; the row's map entry
        // is claimed first, so a row two requests share is placed once (the other
        // ticket's slot stays reserved and the recall returns it)
        const int base_w = __shfl_sync(0xffffffffu, base, __ffs(cmask) - 1);  // cmask != 0 here
        res_full = base_w + __popc(cmask) >= res_len;
        if (cand) {
          const int ticket = base_w + __popc(cmask & ((1u << lane) - 1));
          if (ticket < res_len) {
            const int32_t s = __ldg(P.reserve + ticket);
            if (s >= 0 && s < P.n_g && atomicCAS(P.host_to_gpu + h, kInf, s) == kInf) dst = s;
          } else if (ticket == res_len) {
            set_status(P.status, ECHO_DEV_PREFETCH_CAP_HIT);
          }
        }
      } else if (cand) {
        base = __shfl_sync(grp, base, leader);
        const int ticket = base + __popc(grp & ((1u << lane) - 1));
        const int L = clamp_ctx(__ldg(P.ctx_len + b), P.L_max);
        int cap = (L + P.cap_div - 1) / P.cap_div;
        cap = cap < P.stage_stride ? cap : P.stage_stride;
        if (ticket < cap) {
          dst = b * P.stage_stride + ticket;
        } else if (ticket == cap) {
          set_status(P.status, ECHO_DEV_PREFETCH_CAP_HIT);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kPfRowsPerBatch; ++r) dr[r] = __shfl_sync(0xffffffffu, dst, sl[r]);
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int idx = m * 32 + lane;
      const int r = idx / kKvChunks, c = idx % kKvChunks;
      const int32_t d = pick_reg(dr, r);
      if (r < cnt && d >= 0) dst_rows[static_cast<size_t>(d) * kKvChunks + c] = buf[m];
    }
  }
  if (dst >= 0) {
    if (direct) {  // the row is resident from here on (its bytes are stored above)
      P.to_host[dst] = h;
      P.prio[dst] = kPrefetchedPrio;
    } else {
      P.stage_host[dst] = h;
    }
  }
}

}  // namespace echo
