"""Host logic of the LLM-42 selective-determinism scheduler, on the CPU:
a fake engine and fake fast path built on a Markov "model" whose next token
is a function of (input token, position).  The invariant path is that
function; the fast path deviates from it at some (token, position) pairs.
Flagged requests must end with exactly the invariant sequence (every token
verified, the verifier's token continuing after a rollback); unflagged ones
keep the fast path's tokens; positions, windows and commits are checked
against the model."""
import numpy as np
import torch

V = 1009


def nxt(x, pos):
    return (int(x) * 7919 + int(pos) * 104729 + 17) % V


def fast_tok(x, pos):
    t = nxt(x, pos)
    return (t + 1) % V if (int(x) + int(pos)) % 7 == 0 else t


class FakeShape:
    vocab = V


class FakeEngine:
    device = "cpu"
    shape = FakeShape()

    def __init__(self):
        self.reserved = {}
        self.calls = []

    def reserve(self, slot, n):
        self.reserved[slot] = max(self.reserved.get(slot, 0), n)

    def verify(self, slots, kv_lens, last_tokens, windows, logits=None):
        commit, fix = [], []
        for s, kv, last, w in zip(slots, kv_lens, last_tokens, windows):
            x, j, f = last, len(w), -1
            for i, c in enumerate(w):
                v = nxt(x, kv + i)
                if v != c:
                    j, f = i, v
                    break
                x = c
            commit.append(j)
            fix.append(f)
            assert self.reserved[s] >= kv + 1
        self.calls.append((list(slots), list(kv_lens), [len(w) for w in
                                                         windows]))
        return (len(slots), np.array(commit, np.int32),
                np.array(fix, np.int32), np.zeros(0, np.int32))


class FakeFast:
    def __init__(self):
        self.rows = []

    def decode(self, tok, pos, slots, ids, max_kv_len):
        for i in range(tok.numel()):
            ids[i] = fast_tok(tok[i].item(), pos[i].item())
            self.rows.append((slots[i].item(), tok[i].item(), pos[i].item()))
        assert max_kv_len == int(pos.max().item()) + 1


def invariant_continuation(history, n):
    out, x, p = [], history[-1], len(history) - 1
    for _ in range(n):
        x = nxt(x, p)
        out.append(x)
        p += 1
    return out


def test_selective_scheduler_bookkeeping():
    from deterministic_invariant_bf16_gb300 import scheduler
    rng = np.random.default_rng(3)
    eng, fast = FakeEngine(), FakeFast()
    sch = scheduler.SelectiveScheduler(eng, fast, window=8)
    R, max_new = 10, 30
    hist = {}
    for r in range(R):
        h = [int(t) for t in rng.integers(0, V, size=int(rng.integers(3, 40)))]
        hist[r] = h
        sch.adopt(r, h, deterministic=r % 3 != 0, max_new=max_new)
    sch.run()
    out = sch.outputs()
    for r in range(R):
        assert len(out[r]) == max_new
        if r % 3 != 0:
            assert out[r] == invariant_continuation(hist[r], max_new)
        else:
            x, p, want = hist[r][-1], len(hist[r]) - 1, []
            for _ in range(max_new):
                x = fast_tok(x, p)
                want.append(x)
                p += 1
            assert out[r] == want
    st = sch.stats
    assert st["rollbacks"] > 0
    # verify batches respect the fixed 256-row shape and windows <= 8
    for slots, kv, wl in eng.calls:
        assert sum(wl) <= 256 and max(wl) <= 8 and len(set(slots)) == len(
            slots)
    # every fast-path row sits at the request's next position: the input
    # token is the one at that position of the final sequence
    seq = {r: hist[r] + out[r] for r in range(R)}
    for slot, tok, pos in fast.rows:
        assert pos < len(seq[slot]) and seq[slot][pos] == tok or \
            slot % 3 != 0


def test_scheduler_waits_for_verification_at_the_budget():
    """A flagged request never runs ahead of its output budget: candidates
    stop at max_new and the pending window is verified even if short."""
    from deterministic_invariant_bf16_gb300 import scheduler
    eng, fast = FakeEngine(), FakeFast()
    sch = scheduler.SelectiveScheduler(eng, fast, window=32)
    sch.adopt(0, [5, 6, 7], deterministic=True, max_new=5)
    sch.run()
    assert sch.outputs()[0] == invariant_continuation([5, 6, 7], 5)
    assert all(max(wl) <= 5 for _, _, wl in eng.calls)
