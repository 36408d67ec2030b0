// Refresh schedule of the decode loop: host code, no GPU work.
//
// [Polestar §2.A, schedule]: the drift refresh runs selectively, once enough
// tokens have been decoded since the last one (tau_upd), and periodic full
// passes cover positions outside the top-k clusters.  The decision is taken
// on the host after each decode step, from the number of tokens that step
// committed and whether the current block is decided; see polestar.h for the
// rule and the action flags.
#include <climits>

#include "polestar.h"

extern "C" int ps_schedule_step(const ps_schedule_params* p, ps_schedule_state* s,
                                int committed, int block_done) {
  if (p == nullptr || s == nullptr) return -PS_ERR_ARG;
  if (p->tau_upd < 0 || p->full_period < 0 || p->block_len < 1 || committed < 0 ||
      s->since < 0 || s->refreshes < 0 || s->block_start < 0)
    return -PS_ERR_ARG;
  // saturating: a long run without a refresh cannot wrap the count
  s->since = committed > INT_MAX - s->since ? INT_MAX : s->since + committed;
  if (block_done) {
    if (s->block_start > INT_MAX - p->block_len) return -PS_ERR_ARG;
    s->block_start += p->block_len;
    s->since = 0;
    s->refreshes = 0;
    return PS_SCHED_REFRESH | PS_SCHED_FULL | PS_SCHED_SLIDE | PS_SCHED_REINIT;
  }
  if (s->since < p->tau_upd) return 0;
  s->since = 0;
  s->refreshes = s->refreshes == INT_MAX ? 1 : s->refreshes + 1;
  int act = PS_SCHED_REFRESH;
  if (p->full_period > 0 && s->refreshes % p->full_period == 0) act |= PS_SCHED_FULL;
  return act;
}
