"""The refresh schedule of the decode loop (oracle).

Test infrastructure: only tests/ use this module; it shares no code with the
library.

[Polestar §2.A, schedule]: updates are triggered selectively, once the
decoded context has moved enough (for example after tau_upd tokens have been
decoded), or by periodic full passes over positions outside the local
window.  The page gives no further rule; the reading taken, decided after
each decode step for the next one:

* committed tokens accumulate in `since`; once since >= tau_upd a refresh
  runs (tau_upd = 0: every step) and `since` restarts at 0;
* every full_period-th refresh (full_period > 0) refreshes the whole window
  instead of the top-k clusters' positions;
* when the current block is decided the window slides by one block: the
  next step clusters the new window from scratch (k-means++), refreshes all
  of it, and the counts restart.

Actions (bit flags, as the library's ps_schedule_step returns them):
REFRESH 1, FULL 2, SLIDE 4, REINIT 8.
"""

REFRESH, FULL, SLIDE, REINIT = 1, 2, 4, 8


class ScheduleState:
    def __init__(self):
        self.since = 0        # tokens committed since the last refresh
        self.refreshes = 0    # refreshes since the window was built
        self.block_start = 0  # first position of the current block


def schedule_step(tau_upd, full_period, block_len, state, committed, block_done):
    """Actions of the next step after a step that committed `committed`
    tokens (block_done: the current block has no undecided token left)."""
    state.since += committed
    if block_done:
        state.block_start += block_len
        state.since = 0
        state.refreshes = 0
        return REFRESH | FULL | SLIDE | REINIT
    if state.since < tau_upd:
        return 0
    state.since = 0
    state.refreshes += 1
    act = REFRESH
    if full_period > 0 and state.refreshes % full_period == 0:
        act |= FULL
    return act


def block_progress(commit, undecided, role, current_role=0):
    """The decode loop's outcome of one step, which the schedule above
    consumes: (tokens committed, block decided).  A batch decodes in
    lockstep, so the count is the largest over the batch's sequences of the
    number of positions that committed in this step (every role), and the
    block is decided when no sequence has an undecided position of the
    current block.  commit, undecided: [B][P] flags; role: [P]."""
    B = len(commit)
    committed = 0
    still_open = False
    for b in range(B):
        n = 0
        for j in range(len(role)):
            if commit[b][j]:
                n += 1
            if undecided[b][j] and role[j] == current_role:
                still_open = True
        committed = max(committed, n)
    return committed, not still_open
