// Ring order of a K/V tile pipeline, shared by the warp that fills the
// shared-memory stages and the warps that consume them in the same order.
#pragma once

namespace qpkv {

// K tiles run up to maxlead tiles ahead of V tiles and at most one work
// item ahead; every party walking the schedule sees the same stage order.
struct RingSched {
  int ko, kj, vo, vj, lead;
  int ntl0, ntl1;   // tiles of the items in flight, by parity
  bool kdone;
  int maxlead;
  __device__ __forceinline__ int ntl(int o) const { return (o & 1) ? ntl1 : ntl0; }
  __device__ __forceinline__ void set_ntl(int o, int n) {
    if (o & 1) ntl1 = n; else ntl0 = n;
  }
};
enum : int { kStepK = 0, kStepV = 1, kStepDone = 2, kStepFail = 3 };

// open(o) waits until item o is published and returns its tile count, 0 at
// the end of the work, -1 on failure.
template <class Open>
__device__ __forceinline__ int ring_next(RingSched& q, Open&& open) {
  if (q.vj == q.ntl(q.vo) && q.vo < q.ko) {
    ++q.vo;
    q.vj = 0;
  }
  if (!q.kdone && q.lead < q.maxlead) {
    if (q.kj < q.ntl(q.ko)) return kStepK;
    if (q.ko == q.vo) {
      const int n = open(q.ko + 1);
      if (n < 0) return kStepFail;
      if (n == 0) {
        q.kdone = true;
      } else {
        ++q.ko;
        q.kj = 0;
        q.set_ntl(q.ko, n);
        return kStepK;
      }
    }
  }
  return q.vj < q.ntl(q.vo) ? kStepV : kStepDone;
}

}  // namespace qpkv
