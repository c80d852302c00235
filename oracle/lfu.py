"""Reference policy of the per-layer expert-slot pool.  TEST INFRASTRUCTURE.

Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
section "Streaming without touching a single GPU kernel": each MoE layer owns a
pool of N expert slots and a small slot-id tensor; when the router names the
experts of the next token, an LFU cache decides which are already resident
(hits), misses are loaded into their assigned slots, and the slot indices are
written into the slot-id tensor before the expert matmul runs.

The page does not spell out the policy.  Plain reading used here:

* every requested expert's use count goes up by one per request (hits too);
* hits keep their slot;
* misses are placed in the order of the request list: the lowest-index free
  slot first, otherwise the slot whose resident expert is not requested by
  the current token and has the lowest use count; ties go to the least
  recently used slot, then to the lowest slot index;
* an expert named twice in one request gets one slot;
* a request may name at most ``num_slots`` distinct experts.

The policy only changes hit rate and copy volume; whatever it picks, the
expert matmul through the pool must equal the matmul on the full tensor.
"""

from __future__ import annotations


class LFUSlotPoolRef:
    def __init__(self, num_experts: int, num_slots: int):
        if num_experts < 1 or num_slots < 1:
            raise ValueError("need at least one expert and one slot")
        self.num_experts = num_experts
        self.num_slots = num_slots
        self.count = [0] * num_experts
        self.expert_in_slot = [-1] * num_slots
        self.slot_of_expert = {}
        self.last_use = [-1] * num_slots
        self.step_no = 0

    def step(self, ids):
        """Remap one request.  Returns (slot_ids, misses), misses = [(expert, slot)]."""
        ids = [int(e) for e in ids]
        for e in ids:
            if not 0 <= e < self.num_experts:
                raise ValueError(f"expert id {e} out of range")
        needed = set(ids)
        if len(needed) > self.num_slots:
            raise ValueError("more distinct experts requested than slots")
        t = self.step_no
        for e in ids:
            self.count[e] += 1
        slot_ids = [None] * len(ids)
        for i, e in enumerate(ids):
            s = self.slot_of_expert.get(e)
            if s is not None:
                slot_ids[i] = s
                self.last_use[s] = t
        misses = []
        for i, e in enumerate(ids):
            if slot_ids[i] is not None:
                continue
            s = self.slot_of_expert.get(e)     # loaded earlier in this request
            if s is None:
                free = [j for j in range(self.num_slots) if self.expert_in_slot[j] < 0]
                if free:
                    s = free[0]
                else:
                    cands = [j for j in range(self.num_slots)
                             if self.expert_in_slot[j] not in needed]
                    s = min(cands, key=lambda j: (self.count[self.expert_in_slot[j]],
                                                  self.last_use[j], j))
                    del self.slot_of_expert[self.expert_in_slot[s]]
                self.expert_in_slot[s] = e
                self.slot_of_expert[e] = s
                misses.append((e, s))
            self.last_use[s] = t
            slot_ids[i] = s
        self.step_no += 1
        return slot_ids, misses
