"""Continuous-batching scheduler model (test infrastructure only).

What it follows:
* [LLM-INF] 3.1 (iteration-level batching): after every iteration finished
  requests leave the batch and give back their memory, and waiting requests
  join it;
* [KV-CB] 三, the ContinuousBatchScheduler sketch: running requests are kept,
  then waiting requests fill the batch up to max_batch_size while the KV
  budget allows; a request that does not fit goes back to the head of the
  queue and admission stops (first come, first served, [LLM-INF] 3.3);
* [KV-CB] 4.1 (chunked prefill): prompts are cut into chunks that share an
  iteration with decode steps, under a per-iteration token budget;
* [LLM-INF] 3.2 (preemption and restore): when memory runs short the request
  holding the most pages is written out to host memory (or, when that is
  full, dropped and recomputed later); it is read back when memory is free.

Readings where the sketch is incomplete or wrong (each listed with the design
notes):
* the KV budget is the block manager's live free-block count, so every
  admission lowers it (the sketch checks each request against the same
  stale number);
* decode steps of running requests come first: their appends are reserved
  before anything else, preempting while they do not fit; they run even
  when they use up the token budget, which only limits prefill tokens;
* then running requests with prompt tokens left continue their prefill, in
  batch order, then waiting requests are admitted in arrival order; a chunk
  is the smaller of the prompt tokens left, the token budget left and (for
  a continuing request) the room its blocks plus the free blocks give;
  admission stops at the first request whose first chunk does not fit;
* the iteration that prefills the last prompt token produces the first
  output token; every later iteration appends the previous output token's
  K/V (one slot) and produces the next; a request with max_new outputs is
  finished when the max_new-th is produced and leaves at the next step;
* preemption: the running request holding the most blocks (the later
  arrival on a tie) is swapped to the host pool, its blocks in logical order
  to host blocks taken from the host free list front, when the host pool
  has room for it; otherwise the running request holding the fewest blocks
  (the later arrival on a tie) is dropped -- the page drops shorter
  sequences -- its blocks are released and it goes back to the waiting
  queue to start over (prompt and outputs recomputed).  Dropping the
  largest instead lets the request that needs a block drop itself and lose
  its progress, alternately with another, forever;
* swapped requests come back after the running requests' prefill chunks
  and before new admissions, in arrival order, when their blocks fit and
  the batch has room (a running prefill that waits for blocks would
  otherwise lose them to a returning request again and again); they take
  part again from the
  next iteration (the copy back is ordered before that iteration's kernels);
  a request preempted in an iteration comes back (or is re-admitted) in a
  later one at the earliest, and it holds back the ones queued behind it
  (otherwise the request that needs a block can be its own victim, leave and
  return in the same iteration, forever);
* an iteration in which nothing could be scheduled while requests are
  running (prefills that all wait for blocks) preempts one victim, so the
  others can progress;
* a request that could not complete alone in the pool
  (ceil((prompt + max_new) / 16) > num_blocks) is refused when added.
"""
from collections import deque

from .allocator import BlockAllocator, InvalidOp, blocks_for, BLOCK_SIZE

WAITING, PREFILL, DECODE, SWAPPED, FINISHED = range(5)


class Request:
    def __init__(self, rid, prompt, max_new, arrival):
        self.id, self.prompt, self.max_new, self.arrival = rid, prompt, max_new, arrival
        self.state = WAITING
        self.prefilled = 0      # prompt tokens whose K/V are in the cache
        self.generated = 0      # output tokens produced
        self.resume = None      # state to return to after a swap
        self.host = []          # host blocks while swapped
        self.out_at = -1        # iteration it was last preempted

    def ctx(self):
        """Tokens whose K/V the cache holds."""
        return self.prefilled + max(0, self.generated - 1)


class StepResult:
    def __init__(self):
        self.items = []       # (id, kind "prefill"/"decode", start position, slots)
        self.finished = []    # ids retired at the start of the step
        self.swap_out = []    # (gpu block, host block)
        self.swap_in = []     # (host block, gpu block)
        self.recomputed = []  # ids dropped back to the waiting queue


class Scheduler:
    def __init__(self, num_blocks, max_batch, max_tokens, host_blocks, free_order=None):
        if max_batch <= 0 or max_tokens <= 0 or host_blocks < 0:
            raise InvalidOp("max_batch, max_tokens must be > 0 and host_blocks >= 0")
        self.alloc = BlockAllocator(num_blocks, free_order)
        self.max_batch, self.max_tokens = max_batch, max_tokens
        self.host_total = host_blocks
        self.host_free = deque(range(host_blocks))
        self.waiting, self.running, self.swapped = [], [], []
        self.reqs = {}
        self.arrivals = 0
        self.iteration = 0

    # -- requests ------------------------------------------------------------------
    def add(self, rid, prompt, max_new):
        if rid in self.reqs:
            raise InvalidOp("request id in use")
        if prompt < 1 or max_new < 1:
            raise InvalidOp("prompt and max_new must be >= 1")
        if blocks_for(prompt + max_new) > self.alloc.total:
            raise InvalidOp("request cannot complete in the pool")
        r = Request(rid, prompt, max_new, self.arrivals)
        self.arrivals += 1
        self.reqs[rid] = r
        self.waiting.append(r)

    def idle(self):
        return not (self.waiting or self.running or self.swapped)

    @staticmethod
    def _insert_by_arrival(queue, r):
        i = 0
        while i < len(queue) and queue[i].arrival < r.arrival:
            i += 1
        queue.insert(i, r)

    # -- preemption ------------------------------------------------------------------
    def _preempt(self, out):
        """Swap out the largest running request, or drop the smallest."""
        held = lambda r: len(self.alloc.tables[r.id])
        v = max(self.running, key=lambda r: (held(r), r.arrival))
        if held(v) > len(self.host_free):
            v = min(self.running, key=lambda r: (held(r), -r.arrival))
        tab = self.alloc.tables[v.id]
        self.running.remove(v)
        v.out_at = self.iteration - 1
        if len(tab) <= len(self.host_free):
            v.host = [self.host_free.popleft() for _ in tab]
            out.swap_out.extend(zip(tab, v.host))
            self.alloc.free_seq(v.id)
            v.resume, v.state = v.state, SWAPPED
            self._insert_by_arrival(self.swapped, v)
        else:
            self.alloc.free_seq(v.id)
            v.prefilled = v.generated = 0
            v.state = WAITING
            self._insert_by_arrival(self.waiting, v)
            out.recomputed.append(v.id)

    def _decode_need(self):
        rc = list(self.alloc.refcount)
        return sum(self.alloc._append_need(r.id, rc) for r in self.running if r.state == DECODE)

    # -- one iteration ---------------------------------------------------------------------
    def _finish_chunk(self, r):
        if r.prefilled == r.prompt:
            r.state, r.generated = DECODE, 1
            if r.max_new == 1:
                r.state = FINISHED

    def step(self):
        out = StepResult()
        it = self.iteration
        self.iteration += 1
        # retire
        for r in [r for r in self.running if r.state == FINISHED]:
            self.alloc.free_seq(r.id)
            self.running.remove(r)
            del self.reqs[r.id]
            out.finished.append(r.id)
        # reserve the decode appends
        while self.running and self._decode_need() > len(self.alloc.free):
            self._preempt(out)
        # decodes
        n_dec = 0
        for r in self.running:
            if r.state != DECODE:
                continue
            start = r.ctx()
            slot, _, _ = self.alloc.append_slot(r.id)
            out.items.append((r.id, "decode", start, [slot]))
            r.generated += 1
            if r.generated == r.max_new:
                r.state = FINISHED
            n_dec += 1
        budget = max(0, self.max_tokens - n_dec)
        # prefill continuation
        for r in self.running:
            if r.state != PREFILL or budget == 0:
                continue
            room = len(self.alloc.tables[r.id]) * BLOCK_SIZE - r.ctx() + len(self.alloc.free) * BLOCK_SIZE
            chunk = min(r.prompt - r.prefilled, budget, room)
            if chunk <= 0:
                continue
            start = r.ctx()
            slots, _ = self.alloc.append_tokens(r.id, chunk)
            out.items.append((r.id, "prefill", start, slots))
            r.prefilled += chunk
            budget -= chunk
            self._finish_chunk(r)
        # swapped requests back, before new admissions
        while self.swapped and len(self.running) < self.max_batch:
            v = self.swapped[0]
            if v.out_at == it or blocks_for(v.ctx()) > len(self.alloc.free):
                break
            self.swapped.pop(0)
            self.alloc.alloc_seq(v.id, v.ctx())
            out.swap_in.extend(zip(v.host, self.alloc.tables[v.id]))
            self.host_free.extend(v.host)
            v.host, v.state = [], v.resume
            self.running.append(v)
        # admissions, first come first served
        while self.waiting and len(self.running) < self.max_batch and budget > 0:
            r = self.waiting[0]
            chunk = min(r.prompt, budget)
            if r.out_at == it or blocks_for(chunk) > len(self.alloc.free):
                break
            self.waiting.pop(0)
            self.alloc.alloc_seq(r.id, 0)
            slots, _ = self.alloc.append_tokens(r.id, chunk)
            out.items.append((r.id, "prefill", 0, slots))
            r.prefilled, r.state = chunk, PREFILL
            budget -= chunk
            self._finish_chunk(r)
            self.running.append(r)
        # nothing could run: make room for the others
        if not out.items and not out.swap_in and not out.swap_out and len(self.running) > 1:
            self._preempt(out)
        return out

    # -- invariants (checked by the tests after every step) ---------------------------------
    def check_invariants(self):
        self.alloc.check_invariants()
        held = sum(len(r.host) for r in self.swapped)
        assert held + len(self.host_free) == self.host_total, "host blocks lost"
        assert len(set(self.host_free)) == len(self.host_free)
        assert len(self.running) <= self.max_batch
        for r in self.running:
            assert r.state in (PREFILL, DECODE, FINISHED)
            assert self.alloc.ntokens[r.id] == r.ctx(), "cache tokens != request progress"
        for r in self.swapped:
            assert r.state == SWAPPED and r.id not in self.alloc.tables
            assert len(r.host) == blocks_for(r.ctx())
        for r in self.waiting:
            assert r.state == WAITING and r.id not in self.alloc.tables
        live = {r.id for r in self.running} | {r.id for r in self.swapped} | {r.id for r in self.waiting}
        assert live == set(self.reqs), "a request is lost or duplicated"
        assert set(self.alloc.tables) == {r.id for r in self.running}
