"""Plant plausible mistakes in a private copy of the oracle (CPU only) and
check that at least one pin catches each. The real oracle is untouched."""
import importlib.util
import math
import os

import numpy as np
import pytest

from tests import oracle_pins

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "moe_oracle.py")


def fresh_oracle(tag):
    spec = importlib.util.spec_from_file_location(f"_planted_oracle_{tag}", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def m_nibble_swap(o):
    orig = o.unpack_codes
    def bad(p):
        q = orig(p)
        q2 = q.copy()
        q2[:, 0::2], q2[:, 1::2] = q[:, 1::2], q[:, 0::2]
        return q2
    o.unpack_codes = bad


def m_drop_zero(o):
    def bad(packed, scale, zero, group):
        return o.dequantize.__wrapped__(packed, scale, np.zeros_like(zero), group)
    bad.__wrapped__ = o.dequantize
    o.dequantize = bad


def m_group_mod(o):
    def bad(packed, scale, zero, group):
        q = o.unpack_codes(packed)
        s = np.asarray(scale, np.float64); z = np.asarray(zero, np.float64)
        w = np.empty(q.shape)
        ng = s.shape[1]
        for c in range(q.shape[1]):
            gi = c % ng
            w[:, c] = (q[:, c] - z[:, gi]) * s[:, gi]
        return w
    o.dequantize = bad


def m_tie_high(o):
    orig = o.route
    def bad(logits, k, renorm):
        lg = np.asarray(logits, np.float32)[:, ::-1].copy()
        ids, w = orig(lg, k, renorm)
        return (lg.shape[1] - 1 - ids).astype(np.int32), w
    o.route = bad


def m_always_renorm(o):
    orig = o.route
    o.route = lambda logits, k, renorm: orig(logits, k, True)


def m_never_renorm(o):
    orig = o.route
    o.route = lambda logits, k, renorm: orig(logits, k, False)


def m_ascending(o):
    orig = o.route
    def bad(logits, k, renorm):
        return orig(-np.asarray(logits, np.float32), k, renorm)
    o.route = bad


def m_silu_sign(o):
    o.silu = lambda v: v / (1.0 + np.exp(v))


def m_swap_gate_up(o):
    def bad(x, wg, wu, wd):
        x = np.asarray(x, np.float64)
        return wd @ (o.silu(wu @ x) * (wg @ x))
    o.expert_ffn = bad


def m_transposed_down(o):
    def bad(x, wg, wu, wd):
        x = np.asarray(x, np.float64)
        h = o.silu(wg @ x) * (wu @ x)
        return wd.T[:, :h.shape[0]].T @ h if wd.shape[0] != wd.shape[1] else wd.T @ h
    o.expert_ffn = bad


def m_drop_weight(o):
    orig = o.route
    def bad(logits, k, renorm):
        ids, w = orig(logits, k, renorm)
        return ids, np.ones_like(w)
    o.route = bad


def m_unstable_sort(o):
    orig = o.token_sort
    def bad(ids, E):
        off, pt, pj = orig(ids, E)
        for e in range(E):
            a, b = off[e], off[e + 1]
            pt[a:b] = pt[a:b][::-1].copy(); pj[a:b] = pj[a:b][::-1].copy()
        return off, pt, pj
    o.token_sort = bad


def m_victim_max(o):
    cls = o.ResidencyLayer
    orig_min = min
    class Bad(cls):
        def step(self, needed):
            import builtins
            saved = builtins.min
            def fake_min(it, key=None, **kw):
                if key is not None:
                    return max(it, key=key)
                return saved(it, **kw) if not kw else saved(it, **kw)
            o.min = fake_min
            try:
                return cls.step(self, needed)
            finally:
                del o.min
    o.ResidencyLayer = Bad


def m_decay_after_bump(o):
    cls = o.ResidencyLayer
    class Bad(cls):
        def step(self, needed):
            d = self.decay
            self.decay = 1.0
            out = cls.step(self, needed)
            self.decay = d
            self.counts = [c * d for c in self.counts]
            return out
    o.ResidencyLayer = Bad


def m_coverage_formula(o):
    o.expected_touched = lambda E, k, n: E * (1.0 - (1.0 - k / E) ** (n + 1))


def m_time_model_no_compute(o):
    o.time_model = lambda t_calc, bytes_out, bandwidth: bytes_out / bandwidth


def m_fit_slope_as_bandwidth(o):
    orig = o.fit_time_model
    def bad(b, t):
        tc, bw = orig(b, t)
        return tc, 1.0 / bw
    o.fit_time_model = bad


def m_outside_counts_resident(o):
    o.expected_outside = lambda E, C, k, n: C * (1.0 - (1.0 - k / E) ** n)


def m_prefetch_keeps_unused(o):
    cls = o.ResidencyLayer
    class Bad(cls):
        def step(self, needed):
            keep = {e: sl for e, sl in self.staged.items() if e not in set(int(x) for x in needed)}
            out = cls.step(self, needed)
            for e, sl in keep.items():  # unused staged copies are not freed
                self.free.remove(sl)
            return out
    o.ResidencyLayer = Bad


def m_prefetch_ignores_staged(o):
    cls = o.ResidencyLayer
    class Bad(cls):
        def step(self, needed):
            self.free.extend(self.staged.values())  # staged misses copied again into a free slot
            self.staged = {}
            return cls.step(self, needed)
    o.ResidencyLayer = Bad


MUTATIONS = [m_nibble_swap, m_drop_zero, m_group_mod, m_tie_high, m_always_renorm,
             m_never_renorm, m_ascending, m_silu_sign, m_swap_gate_up,
             m_transposed_down, m_drop_weight, m_unstable_sort, m_victim_max,
             m_decay_after_bump, m_coverage_formula, m_time_model_no_compute,
             m_fit_slope_as_bandwidth, m_outside_counts_resident, m_prefetch_keeps_unused,
             m_prefetch_ignores_staged]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutation):
    o = fresh_oracle(mutation.__name__)
    mutation(o)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except Exception:  # AssertionError, or a shape/arith error it provokes
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutation.__name__}"
