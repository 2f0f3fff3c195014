// Greedy damage-per-byte bitwidth planner (host code).
//
// PagedWeight, "Core components" 2 (quality-aware runtime planner): each
// possible bitwidth cut gets a damage score; when a memory target is set the
// planner takes the cuts with the least damage per byte saved, greedily.
// Frequently routed ("hot") experts are protected by a higher bitwidth floor
// and a damage multiplier.  The pages give no formulas; the ones here (the
// 4^-b error model, m_e = max(1, E * share_e), hot = share above 1/E) are the
// plainest reading and are stated in include/pw.h.
//
// Each block holds at most one live candidate (its next rung down), kept in a
// priority queue ordered by damage per byte, then block id; taking a cut
// queues the block's next one.  A block's successive cuts cost more per byte
// (4^-b is convex along the ladder), so the cuts are taken in non-decreasing
// order of damage per byte.
#include <cstdint>
#include <queue>
#include <vector>

#include "pw_internal.cuh"

namespace pw {
namespace {

const int kLadder[5] = {3, 4, 5, 6, 8};

int rung_of(int q) {
  for (int i = 0; i < 5; ++i)
    if (kLadder[i] == q) return i;
  return -1;
}

double quant_error(int b) { return 1.0 / static_cast<double>(1ull << (2 * b)); }   // 4^-b

struct Cut {
  double ratio;    // damage per byte saved
  int32_t block;
  int to;          // bitwidth after the cut
  int64_t bytes;   // bytes the cut saves
};

struct CutOrder {  // min-heap on (ratio, block)
  bool operator()(const Cut& x, const Cut& y) const {
    if (x.ratio != y.ratio) return x.ratio > y.ratio;
    return x.block > y.block;
  }
};

}  // namespace
}  // namespace pw

extern "C" int pw_plan_recommit(int32_t n_blocks, const int32_t* q_now, const float* sensitivity,
                                const int64_t* bytes_per_bit, const float* routing_mass,
                                int32_t hot_floor, int64_t bytes_to_free, int32_t* out_ids,
                                int32_t* out_q, int32_t* n_out, int64_t* bytes_freed) {
  using namespace pw;
  if (n_blocks < 0 || n_blocks % 2)
    return fail(PW_ERR_INVALID_ARG, "n_blocks (%d) must be even and >= 0", n_blocks);
  if (!n_out || !bytes_freed) return fail(PW_ERR_INVALID_ARG, "NULL output pointer");
  *n_out = 0;
  *bytes_freed = 0;
  if (n_blocks == 0) return PW_OK;
  if (!q_now || !sensitivity || !bytes_per_bit || !routing_mass || !out_ids || !out_q)
    return fail(PW_ERR_INVALID_ARG, "NULL pointer");
  if (rung_of(hot_floor) < 0) return fail(PW_ERR_UNSUPPORTED_Q, "hot_floor %d off the ladder", hot_floor);
  const int E = n_blocks / 2;
  double total_mass = 0.0;
  for (int e = 0; e < E; ++e) {
    if (!(routing_mass[e] >= 0.f)) return fail(PW_ERR_INVALID_ARG, "routing_mass[%d] < 0", e);
    total_mass += static_cast<double>(routing_mass[e]);
  }
  std::vector<int> q(n_blocks), floor_q(n_blocks);
  std::vector<double> mult(n_blocks);
  for (int i = 0; i < n_blocks; ++i) {
    if (rung_of(q_now[i]) < 0) return fail(PW_ERR_UNSUPPORTED_Q, "block %d: q %d off the ladder", i, q_now[i]);
    if (!(sensitivity[i] >= 0.f) || bytes_per_bit[i] < 0)
      return fail(PW_ERR_INVALID_ARG, "block %d: negative sensitivity or bytes", i);
    const double m = static_cast<double>(routing_mass[i / 2]);
    const bool hot = total_mass > 0.0 && m * E > total_mass;
    q[i] = q_now[i];
    floor_q[i] = hot ? hot_floor : kLadder[0];
    mult[i] = total_mass > 0.0 ? (m * E / total_mass > 1.0 ? m * E / total_mass : 1.0) : 1.0;
  }
  std::priority_queue<Cut, std::vector<Cut>, CutOrder> heap;
  auto push_next = [&](int i) {
    const int r = rung_of(q[i]);
    if (r <= 0) return;
    const int to = kLadder[r - 1];
    if (to < floor_q[i]) return;
    const int64_t bytes = static_cast<int64_t>(q[i] - to) * bytes_per_bit[i];
    if (bytes <= 0) return;
    const double damage = static_cast<double>(sensitivity[i]) * mult[i] *
                          (quant_error(to) - quant_error(q[i]));
    heap.push(Cut{damage / static_cast<double>(bytes), i, to, bytes});
  };
  for (int i = 0; i < n_blocks; ++i) push_next(i);
  int64_t freed = 0;
  while (freed < bytes_to_free && !heap.empty()) {
    const Cut c = heap.top();
    heap.pop();
    q[c.block] = c.to;
    freed += c.bytes;
    push_next(c.block);
  }
  int n = 0;
  for (int i = 0; i < n_blocks; ++i) {
    if (q[i] != q_now[i]) {
      out_ids[n] = i;
      out_q[n] = q[i];
      ++n;
    }
  }
  *n_out = n;
  *bytes_freed = freed;
  return PW_OK;
}
