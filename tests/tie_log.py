"""Near-tie accounting of the code-parity tests.

A GPU code that differs from the oracle's is accepted only as a near-tie:
the oracle's fp32 distances of the two centroids differ by less than 1e-6
relative.  Every parity check records how many codes it compared, how many
differed as near-ties, how many differed otherwise (must be 0) and, where
the call reported it, the GPU's own near-tie counter (subvectors whose best
two fp32 distances were that close).  The records are printed at the end of
the pytest run (conftest.py, terminal summary), so the counts appear in the
test log whether or not output is captured."""
from __future__ import annotations

RECORDS: list[dict] = []


def bound(n_codes: int) -> float:
    """Largest number of near-tie mismatches accepted in n_codes codes of
    continuous synthetic data: two fp32 distances within 1e-6 relative of
    each other are rare (well under 1e-4 per subvector); a test whose
    centroids tie on purpose does not use this bound."""
    return 2 + 1e-4 * n_codes


def record(name: str, n_codes: int, near_ties: int, fails: int, device_count=None) -> None:
    RECORDS.append(dict(name=name, n_codes=int(n_codes), near_ties=int(near_ties), fails=int(fails),
                        device_count=None if device_count is None else int(device_count)))


def summary_lines() -> list[str]:
    if not RECORDS:
        return []
    tot = sum(r["n_codes"] for r in RECORDS)
    ties = sum(r["near_ties"] for r in RECORDS)
    fails = sum(r["fails"] for r in RECORDS)
    out = [f"{len(RECORDS)} code-parity checks, {tot} codes: {ties} near-tie mismatches, {fails} failing mismatches"]
    for r in RECORDS:
        dev = "" if r["device_count"] is None else f", GPU near-tie counter {r['device_count']}"
        out.append(f"  {r['name']}: {r['n_codes']} codes, {r['near_ties']} near-tie mismatches, "
                   f"{r['fails']} failing{dev}")
    return out
