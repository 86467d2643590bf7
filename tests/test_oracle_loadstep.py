"""The load-step experiment on the oracle: its shape ("Adaptive
DHiSparse", Evidence: with optional residency on, fewer selected rows come
from the host while load is low; the optional pages give way under memory
pressure and come back once the extra requests have left), and the
machinery's invariants at every step."""
import numpy as np

from dhs_workload.loadstep import LOADSTEP_SMALL, phase_fractions, run
from fixture_runner import OracleAdapter


class CheckedOracle(OracleAdapter):
    def resolve(self, step, r, s, sel):
        out = super().resolve(step, r, s, sel)
        assert self.p.check(r, s) == 0
        return out


def test_loadstep_shape(oracle_lib, gen_lib):
    cfg = LOADSTEP_SMALL
    on = run(CheckedOracle(), cfg, residency=True)
    off = run(OracleAdapter(), cfg, residency=False)
    f_on, f_off = phase_fractions(on), phase_fractions(off)
    # residency cuts host fetches at low load ...
    assert f_on["low"] < 0.25 * f_off["low"], (f_on, f_off)
    # ... gives memory up under pressure (host fetches rise) ...
    assert f_on["burst"] > 2 * f_on["low"], f_on
    # ... and repopulates as requests drain
    drain = [x for x in on if x["phase"] == "drain"]
    assert drain[-1]["resident_pages"] == cfg.capacity
    assert drain[-1]["host"] < drain[0]["host"]
    assert f_on["drain"] < f_on["burst"]
    # backups keep up: nothing pending once the burst's admissions are done
    assert on[-1]["pending_backup"] == 0
    # without residency nothing is ever optional-resident
    assert all(x["resident_pages"] == 0 for x in off)


def test_loadstep_pressure_reclaims_oldest_first(oracle_lib, gen_lib):
    cfg = LOADSTEP_SMALL
    seen = {}

    class Spy(OracleAdapter):
        def reclaim(self, order, deficit):
            rc, freed = super().reclaim(order, deficit)
            seen.setdefault("orders", []).append(list(order))
            return rc, freed

    recs = run(Spy(), cfg, residency=True)
    # every reclaim walks the admitted requests oldest first
    for order in seen["orders"]:
        assert order == sorted(order)
    # at the end of the burst the youngest requests hold the capacity
    burst_end = [x for x in recs if x["phase"] == "burst"][-1]
    assert burst_end["resident_pages"] <= cfg.capacity
