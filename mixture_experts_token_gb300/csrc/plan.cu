// Dynamic redundant experts: the duplication plan.
//
// "Moe dynamic redundancy" (MaxText pull request 4760), review comments on
// plan_expert_duplication: duplicate the hottest not-yet-duplicated expert
// of the most loaded rank (r_max) into a spare slot on an underloaded rank,
// divert part of its tokens there, and stop when r_max has no
// un-duplicated expert left (has_candidate), so that no expert is
// duplicated twice.  Each round here: r_max = most loaded shard, e* = its
// hottest expert with rows and no duplicate, r_min = least loaded other
// shard with a free slot (ties: lower index everywhere); stop when e* or
// r_min is missing or the gap is zero; else move
// n = min(rows of e*, (load[r_max] - load[r_min]) / 2) rows of e* to the
// next free slot of r_min.  Integer arithmetic only, so the plan is exact.
//
// One warp: the argmax/argmin of a round are warp reductions over 64-bit
// keys (value in the high word, complemented index in the low word, so the
// lower index wins ties); the state lives in shared memory.
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__global__ void __launch_bounds__(32) plan_kernel(
    const int32_t* __restrict__ counts, int E, int S, int B, long long cap,
    int32_t* __restrict__ divert_out, int32_t* __restrict__ slot_out,
    int32_t* __restrict__ group_expert, int32_t* __restrict__ shard_after,
    int32_t* __restrict__ flag_after) {
  __shared__ int cnt[kMaxExperts];
  __shared__ int divert[kMaxExperts];
  __shared__ int slot_of[kMaxExperts];
  __shared__ int load[kMaxShards];
  __shared__ int freeslots[kMaxShards];
  const int lane = threadIdx.x;
  const int Es = E / S, Gs = Es + B, G = S * Gs;
  for (int e = lane; e < E; e += 32) {
    cnt[e] = counts[e];
    divert[e] = 0;
    slot_of[e] = -1;
  }
  __syncwarp();
  for (int s = lane; s < S; s += 32) {
    long long sum = 0;
    for (int e = s * Es; e < (s + 1) * Es; ++e) sum += cnt[e];
    load[s] = static_cast<int>(sum);
    freeslots[s] = B;
  }
  __syncwarp();

  for (int round = 0; round < S * B; ++round) {
    // r_max: the most loaded shard
    uint64_t key = 0;
    for (int s = lane; s < S; s += 32) {
      const uint64_t k2 = (static_cast<uint64_t>(load[s]) << 32) |
                          (0xffffffffu - static_cast<uint32_t>(s));
      key = k2 > key ? k2 : key;
    }
    key = warp_max_u64(key);
    const int r_max = static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
    // e*: its hottest expert with rows and no duplicate yet
    uint64_t ek = 0;
    for (int e = r_max * Es + lane; e < (r_max + 1) * Es; e += 32) {
      if (slot_of[e] < 0 && cnt[e] > 0) {
        const uint64_t k2 = (static_cast<uint64_t>(cnt[e]) << 32) |
                            (0xffffffffu - static_cast<uint32_t>(e));
        ek = k2 > ek ? k2 : ek;
      }
    }
    ek = warp_max_u64(ek);
    const bool has_candidate = ek != 0;
    // r_min: the least loaded other shard with a free slot
    uint64_t mk = 0;  // max of the complemented load = min load
    for (int s = lane; s < S; s += 32) {
      if (s != r_max && freeslots[s] > 0) {
        const uint64_t k2 =
            (static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(load[s]))
             << 32) |
            (0xffffffffu - static_cast<uint32_t>(s));
        mk = k2 > mk ? k2 : mk;
      }
    }
    mk = warp_max_u64(mk);
    if (!has_candidate || mk == 0) break;
    const int r_min = static_cast<int>(0xffffffffu - static_cast<uint32_t>(mk));
    const int gap = load[r_max] - load[r_min];
    if (gap <= 0) break;
    const int e_star =
        static_cast<int>(0xffffffffu - static_cast<uint32_t>(ek));
    const int n = min(cnt[e_star], gap / 2);
    if (n <= 0) break;
    __syncwarp();
    if (lane == 0) {
      const int b = B - freeslots[r_min];
      freeslots[r_min] -= 1;
      slot_of[e_star] = r_min * Gs + Es + b;
      divert[e_star] = n;
      load[r_max] -= n;
      load[r_min] += n;
    }
    __syncwarp();
  }

  for (int e = lane; e < E; e += 32) {
    divert_out[e] = divert[e];
    slot_out[e] = slot_of[e];
  }
  for (int g = lane; g < G; g += 32) {
    const int s = g / Gs, q = g % Gs;
    group_expert[g] = q < Es ? s * Es + q : -1;
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32)
    if (slot_of[e] >= 0) group_expert[slot_of[e]] = e;
  int over = 0;
  for (int s = lane; s < S; s += 32) {
    shard_after[s] = load[s];
    if (cap >= 0 && load[s] > cap) over = 1;
  }
  over = __any_sync(0xffffffffu, over);
  if (lane == 0) *flag_after = over;
}

}  // namespace

cudaError_t launch_plan(const moe_config_t& c, const int32_t* counts,
                        int32_t* divert, int32_t* slot_of,
                        int32_t* group_expert, int32_t* shard_after,
                        int32_t* flag_after, cudaStream_t s) {
  plan_kernel<<<1, 32, 0, s>>>(counts, c.E, c.S, c.redundant_slots,
                               capacity_rows(c), divert, slot_of,
                               group_expert, shard_after, flag_after);
  return cudaGetLastError();
}

}  // namespace moe
