"""The oracle's pins catch plausible mistakes.

For each oracle function, a copy of its module with one planted change (a
dropped term, a wrong sign, index or axis, a reversed order, a swapped
operand) is built here on the CPU and run through the pins of that function
(tests/test_oracle_*.py); at least one pin must fail on every copy. The
planted changes exist only in these copies: the oracle itself is untouched.
Changes that leave the result the same (for example writing every miss in
ascending order, when only the last writes per slot survive anyway) are not
mistakes and are not planted.
"""
import pathlib
import types

import pytest

import oracle
import oracle.step
import test_oracle_plan
import test_oracle_reuse
import test_oracle_sfa
import test_oracle_step
import test_oracle_topk
import test_policy_hit_rates

ORACLE = pathlib.Path(oracle.__file__).parent


def mutant(fname: str, old: str, new: str) -> types.ModuleType:
    """The oracle module `fname` with `old` (which must occur exactly once)
    replaced by `new`."""
    src = (ORACLE / fname).read_text()
    assert src.count(old) == 1, f"{fname}: the planted change must match once: {old!r}"
    mod = types.ModuleType(f"mutant_{fname[:-3]}")
    mod.__package__ = "oracle"  # its relative imports resolve to the oracle's modules
    exec(compile(src.replace(old, new), f"<mutant of {fname}>", "exec"), mod.__dict__)
    return mod


def failing_pins(target, patches: dict, pins) -> list:
    """Run the pins (callables) with `patches` applied to `target` (a module
    whose globals the pins read); return the pins that failed."""
    failed = []
    for pin in pins:
        with pytest.MonkeyPatch.context() as mp:
            for name, value in patches.items():
                mp.setattr(target, name, value)
            try:
                pin()
            except (Exception, pytest.fail.Exception):  # an assertion, a pytest.raises
                failed.append(pin)                        # that saw no error, or an error
    return failed


TOPK_PINS = [test_oracle_topk.test_brute_force_tiny_all_k, test_oracle_topk.test_invariants_large,
             test_oracle_topk.test_signed_zero_is_one_score,
             test_oracle_topk.test_all_equal_takes_lowest_positions,
             test_oracle_topk.test_context_bound_and_nan]

TOPK_MUTANTS = {
    "ties go to the higher position": ("np.lexsort((pos, -s))", "np.lexsort((-pos, -s))"),
    "smallest scores selected": ("np.lexsort((pos, -s))", "np.lexsort((pos, s))"),
    "output left in score order": ("np.sort(order[:k])", "order[:k]"),
    "best position dropped": ("np.sort(order[:k])", "np.sort(order[1:k + 1])"),
    "NaN accepted": ("if np.isnan(s).any():", "if False:"),
    "context bound ignored": ("s = np.asarray(scores[:ctx_len]", "s = np.asarray(scores[:len(scores)]"),
}


@pytest.mark.parametrize("what", sorted(TOPK_MUTANTS))
def test_topk_pins_catch(what):
    m = mutant("topk.py", *TOPK_MUTANTS[what])
    assert failing_pins(test_oracle_topk, {"topk_ids": m.topk_ids}, TOPK_PINS), what


PLAN_PINS = [test_oracle_plan.test_hand_worked_overflow, test_oracle_plan.test_duplicates_listed_once,
             test_oracle_plan.test_random_sequences_against_simulator,
             test_oracle_plan.test_hits_plus_misses_is_k_for_distinct_ids,
             test_oracle_plan.test_install_code_orders_installs_around_hit_reads]

PLAN_MUTANTS = {
    "set from the wrong hash": ("        s = t % S\n        way = None",
                                "        s = (t // W) % S\n        way = None"),
    "hit slot index transposed": ("src_map[j] = s * W + way", "src_map[j] = way * S + s"),
    "miss encoded without the offset": ("src_map[j] = -1 - t", "src_map[j] = -t"),
    "last position of a repeated miss": ("first_pos.setdefault(t, j)", "first_pos[t] = j"),
    "misses in descending order": ("miss_ids = sorted(first_pos)",
                                   "miss_ids = sorted(first_pos, reverse=True)"),
    "victim ignores the rank": ("victim.append(s * W + (ptr[s] + r) % W)",
                                "victim.append(s * W + ptr[s] % W)"),
    "one install too few on overflow": ("install.append(r >= count[s] - W)",
                                        "install.append(r > count[s] - W)"),
    "pointer advances by installs only": ("ptr_next = [(ptr[s] + count[s]) % W",
                                          "ptr_next = [(ptr[s] + min(count[s], W)) % W"),
    "installs never wait for the hit reads": (
        "0 if not keep else 2 if int(v) in hit_slots else 1", "0 if not keep else 1"),
}


@pytest.mark.parametrize("what", sorted(PLAN_MUTANTS))
def test_plan_pins_catch(what):
    m = mutant("plan.py", *PLAN_MUTANTS[what])
    assert failing_pins(test_oracle_plan, {"dsa_plan": m.dsa_plan}, PLAN_PINS), what


SFA_PINS = [test_oracle_sfa.test_constant_rows_give_the_row, test_oracle_sfa.test_single_row,
            test_oracle_sfa.test_two_rows_sigmoid_weights,
            test_oracle_sfa.test_row_permutation_invariance_and_zero_scale,
            test_oracle_sfa.test_round_to_bf16_ties_to_even]

SFA_MUTANTS = {
    "scale dropped": ("s = scale * (q @ K.T)", "s = (q @ K.T)"),
    "rope part dropped from the scores": ("s = scale * (q @ K.T)",
                                          "s = scale * (q[:, :D_LATENT] @ K[:, :D_LATENT].T)"),
    "V taken from the row's tail": ("(p @ K[:, :D_LATENT])", "(p @ K[:, -D_LATENT:])"),
    "max over heads": ("m = s.max(axis=1, keepdims=True)", "m = s.max(axis=0, keepdims=True)"),
    "normaliser over heads": ("Z = p.sum(axis=1, keepdims=True)", "Z = p.sum(axis=0, keepdims=True)"),
    "lse without the max": ("lse = m[:, 0] + np.log(Z[:, 0])", "lse = np.log(Z[:, 0])"),
    "rounding truncates": ("r = np.rint(m * 256.0) / 256.0", "r = np.trunc(m * 256.0) / 256.0"),
}


@pytest.mark.parametrize("what", sorted(SFA_MUTANTS))
def test_sfa_pins_catch(what):
    m = mutant("sfa.py", *SFA_MUTANTS[what])
    patches = {"sfa_decode": m.sfa_decode, "round_to_bf16_bits": m.round_to_bf16_bits}
    assert failing_pins(test_oracle_sfa, patches, SFA_PINS), what


STEP_PINS = [test_oracle_step.test_tiny_workload_steps,
             test_oracle_step.test_repeat_step_is_all_hits_without_overflow]

STEP_MUTANTS = {
    "served host row off by one": ("serve.py", "out[j] = host_rows[t]", "out[j] = host_rows[t - 1]",
                                   "dsa_serve"),
    "served pool slot off by one": ("serve.py", "out[j] = pool_rows[src]",
                                    "out[j] = pool_rows[src - 1]", "dsa_serve"),
    "pointers not advanced": ("install.py", "fifo_ptr[:] = plan.ptr_next", "pass",
                              "metadata_update"),
    "refill writes the wrong row": ("install.py", "pool_rows[int(v)] = host_rows[int(t)]",
                                    "pool_rows[int(v)] = host_rows[int(v)]", "dsa_install"),
}


@pytest.mark.parametrize("what", sorted(STEP_MUTANTS))
def test_step_pins_catch(what):
    fname, old, new, name = STEP_MUTANTS[what]
    m = mutant(fname, old, new)
    assert failing_pins(oracle.step, {name: getattr(m, name)}, STEP_PINS), what


def test_reuse_pins_catch():
    m = mutant("reuse.py", "src_map[j] = where[t]", "src_map[j] = j")
    pins = [lambda: test_oracle_reuse.test_against_brute_force(s) for s in range(3)]
    assert failing_pins(test_oracle_reuse, {"plan_reuse": m.plan_reuse}, pins)


def test_lru_pins_catch():
    # no touch of the hits: the pool becomes FIFO by install time
    m = mutant("lru.py", "self.order.move_to_end(t)", "pass")
    pins = [test_policy_hit_rates.test_lru_pool_against_brute_force,
            test_policy_hit_rates.test_lru_special_cases]
    assert failing_pins(oracle, {"LruPool": m.LruPool}, pins)


LRU_SLOT_MUTANTS = {
    "hits not touched": ("                self.last_use[int(src_map[j])] = self.clock", "                pass"),
    "victims in slot order, not least recently used":
        ("key=lambda s: (self.tags[s] >= 0, self.last_use[s], s)",
         "key=lambda s: (self.tags[s] >= 0, s)"),
    "misses installed in descending id": ("miss_ids = sorted(first_pos)",
                                          "miss_ids = sorted(first_pos, reverse=True)"),
}


@pytest.mark.parametrize("name", sorted(LRU_SLOT_MUTANTS))
def test_lru_slot_pins_catch(name):
    old, new = LRU_SLOT_MUTANTS[name]
    m = mutant("lru.py", old, new)
    pins = [test_policy_hit_rates.test_lru_slots_hand_worked] + \
        [lambda a=a: test_policy_hit_rates.test_lru_slots_against_brute_force(*a)
         for a in ((20, 12, 60), (8, 12, 30))]
    assert failing_pins(oracle, {"LruSlots": m.LruSlots}, pins), name


def test_unchanged_copies_pass_every_pin():
    """The harness itself: copies with no change pass all the pins."""
    same = {f: mutant(f, "import numpy as np", "import numpy as np")
            for f in ("topk.py", "plan.py", "sfa.py")}
    assert not failing_pins(test_oracle_topk, {"topk_ids": same["topk.py"].topk_ids}, TOPK_PINS)
    assert not failing_pins(test_oracle_plan, {"dsa_plan": same["plan.py"].dsa_plan}, PLAN_PINS)
    assert not failing_pins(test_oracle_sfa, {"sfa_decode": same["sfa.py"].sfa_decode}, SFA_PINS)
    lru_same = mutant("lru.py", "import numpy as np", "import numpy as np")
    lru_pins = [test_policy_hit_rates.test_lru_slots_hand_worked,
                lambda: test_policy_hit_rates.test_lru_slots_against_brute_force(20, 12, 60)]
    assert not failing_pins(oracle, {"LruSlots": lru_same.LruSlots}, lru_pins)
