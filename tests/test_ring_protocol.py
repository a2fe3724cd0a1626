"""Host-side model of the attention kernel's K/V ring protocol (no GPU).

The kernel's producer warp streams K and V tiles through NSLOT shared-memory
slots in the order K0 V0 K1 V1 ... (load n goes to slot n % NSLOT).  A slot
is reused once the MMAs that read its previous load have completed, which the
kernel learns from release events: event e is relayed by tile 1's softmax
once it saw the commit that follows QK1(e), so every MMA issued before that
commit has completed.  The per-rank instance relays it at the end of the
softmax iteration, after P1(e) is handed over; the sharded instance relays it
as soon as S1(e) is loaded, before P1(e).  The producer waits for
event (n - NSLOT + 1) >> 1 before load n >= NSLOT, on barrier e % NREL with
parity (e // NREL) & 1, NREL = NSLOT // 2 + 1.

The model runs the roles (producer, MMA issuer, the two softmax tiles) as
sequential programs.  Tensor-core work completes as late as the protocol
allows: a commit fires only when no role can otherwise progress.  It checks,
for every key-tile count up to 64, both ring sizes and both relay places, that
- every role finishes (no wait that never ends),
- no load overwrites a slot whose previous load still has an MMA in flight,
- no release barrier runs a whole phase past the one its waiter expects.
A variant that waits for one event too few must trip the second check.
"""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(__file__), "..", "sequence_video_dit_gb300", "csrc", "sp_attn_tc.cu")


def _source():
    with open(SRC, encoding="utf-8") as f:
        return f.read()


def _ring_sizes():
    # NSLOT per head dim, as the kernel's configuration states it
    m = re.search(r"NSLOT = \(D == 64\) \? (\d+) : (\d+);", _source())
    assert m, "ring size expression not found in the kernel source"
    return {64: int(m.group(1)), 128: int(m.group(2))}


def test_model_matches_the_kernel_source():
    src = _source()
    # the rules the model below encodes, as the kernel states them
    assert "constexpr int NREL = NSLOT / 2 + 1;" in src
    assert "const int e = (n - NSLOT + 1) >> 1;" in src
    assert "wait_bounded(&bar_rel[e % NREL], (uint32_t)(e / NREL) & 1u" in src
    assert "auto kslot = [](int j) { return (2 * j) % NSLOT; };" in src
    assert "auto vslot = [](int j) { return (2 * j + 1) % NSLOT; };" in src
    assert "if (!TILED && i == 1 && quarter == 0 && lane == 0) mbar_arrive(&bar_rel[jj % NREL]);" in src
    assert "if (TILED && i == 1 && quarter == 0 && lane == 0) mbar_arrive(&bar_rel[jj % NREL]);" in src


def _mma_program(nkv):
    """The MMA issuer's sequence: waits, MMAs (with the load each reads) and commits,
    in the kernel's order PV0(j) QK0(j+1) PV1(j) QK1(j+1)."""
    prog = [("wait_load", 0), ("mma", 0), ("commit", ("sf", 0)), ("mma", 0), ("commit", ("sf", 1))]
    for j in range(nkv):
        more = j + 1 < nkv
        prog += [("wait_load", 2 * j + 1), ("wait_p", (0, j)), ("mma", 2 * j + 1)]
        if more:
            prog += [("wait_load", 2 * j + 2), ("mma", 2 * j + 2), ("commit", ("sf", 0))]
        else:
            prog += [("commit", ("of", 0))]
        prog += [("wait_p", (1, j)), ("mma", 2 * j + 1)]
        prog += [("mma", 2 * j + 2), ("commit", ("sf", 1))] if more else [("commit", ("of", 1))]
    return prog


def _run(nkv, nslot, early=0, relay_on_load=False):
    """Runs the protocol to its end; `early` > 0 makes the producer wait for
    an event that many steps too early (a broken variant).  relay_on_load:
    tile 1 relays event j when S1(j) arrives and hands P1(j) over only when
    no other role can move (as late as possible)."""
    nrel = nslot // 2 + 1
    n_loads = 2 * nkv
    landed = set()
    slot_of = {}                 # slot -> load currently in it
    last_reader = {}             # load -> issue position of its last MMA so far
    issued = 0                   # issue positions (MMAs and commits)
    pending = []                 # commits issued, not fired: (position, kind)
    completed = 0                # every issue position below this has completed
    fired = {("sf", 0): 0, ("sf", 1): 0, ("of", 0): 0, ("of", 1): 0}
    p_ready = {0: 0, 1: 0}
    events = 0                   # release events relayed so far (in order)
    n = 0                        # producer: next load
    mi = 0                       # MMA issuer: next op
    sm = {0: 0, 1: 0}            # softmax tile i: next iteration
    held = False                 # relay_on_load: tile 1 relayed its event, P1 not handed over yet
    prog = _mma_program(nkv)
    while True:
        moved = False
        while n < n_loads:       # producer
            if n >= nslot:
                e = ((n - nslot + 1) >> 1) - early
                # however late the producer looks, event e + NREL cannot have
                # fired: it follows QK1(e + NREL), which reads load 2(e + NREL),
                # and loads from n on are not issued yet
                assert early or 2 * (e + nrel) >= n, f"event {e + nrel} could alias event {e}"
                if e >= 0 and events <= e:
                    break
                # barrier e % NREL has completed phase e // NREL, not the next one
                assert events <= e + nrel, f"phase alias at load {n} (event {e})"
                old = slot_of[n % nslot]
                assert last_reader.get(old, -1) < completed, f"load {n} overwrites load {old} in use"
            slot_of[n % nslot] = n
            landed.add(n)
            n += 1
            moved = True
        while mi < len(prog):    # MMA issuer
            op, arg = prog[mi]
            if op == "wait_load" and arg not in landed:
                break
            if op == "wait_p" and p_ready[arg[0]] <= arg[1]:
                break
            if op == "mma":
                last_reader[arg] = issued
                issued += 1
            elif op == "commit":
                pending.append((issued, arg))
                issued += 1
            mi += 1
            moved = True
        for i in (0, 1):         # softmax: S_i(j) in, P_i(j) out; tile 1 relays event j
            while sm[i] < nkv and fired[("sf", i)] > sm[i] and not (i == 1 and held):
                if i == 1 and relay_on_load:
                    events += 1
                    held = True
                    moved = True
                    break
                p_ready[i] += 1
                if i == 1:
                    events += 1
                sm[i] += 1
                moved = True
        if moved:
            continue
        if held:                 # nothing else can move: tile 1 hands P1 over
            held = False
            p_ready[1] += 1
            sm[1] += 1
            continue
        if not pending:
            break
        # nothing else can move: the tensor core finishes the oldest commit's work
        pos, kind = pending.pop(0)
        completed = pos + 1
        fired[kind] += 1
    assert n == n_loads, f"producer stuck at load {n} of {n_loads}"
    assert mi == len(prog), f"MMA issuer stuck at op {mi} of {len(prog)}: {prog[mi]}"
    assert sm == {0: nkv, 1: nkv}, f"softmax stuck at {sm}"
    assert fired[("of", 0)] == 1 and fired[("of", 1)] == 1


@pytest.mark.parametrize("relay_on_load", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_ring_protocol_finishes_and_never_overwrites_a_slot_in_use(D, relay_on_load):
    nslot = _ring_sizes()[D]
    for nkv in range(1, 65):
        _run(nkv, nslot, relay_on_load=relay_on_load)


@pytest.mark.parametrize("relay_on_load", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_the_model_catches_a_release_one_event_early(D, relay_on_load):
    nslot = _ring_sizes()[D]
    with pytest.raises(AssertionError, match="in use"):
        for nkv in range(1, 65):
            _run(nkv, nslot, early=1, relay_on_load=relay_on_load)
