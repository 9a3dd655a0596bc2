"""Boundary-band accounting of the parity tests.

The bar for decisions (selected draft, accepted length, emitted token) is bit
equality with the oracle, except for trials the oracle flags inside the
boundary band, where an fp32 implementation may legitimately decide otherwise
than fp64.  Each comparison records here how many trials it checked, how many
fell in the band, of which kinds, and on how many of those the GPU still
agreed with the oracle.  ``tests/conftest.py`` prints the table at the end of
every run, so the counts are visible in a plain ``pytest -q`` log.
"""

KINDS = {1: "accept", 2: "cdf", 4: "select", 8: "resid"}

RECORDS = []


class BandCount(int):
    """The number of boundary-band trials of one comparison (an int, so that
    tests can bound it directly), with the details as attributes: checked
    (trials compared), kinds ({kind: trials}; a trial may count under several
    kinds), band_agree (band trials whose decisions still equal the
    oracle's)."""

    def __new__(cls, n, checked=0, kinds=None, band_agree=0, tag=""):
        obj = super().__new__(cls, n)
        obj.checked = checked
        obj.kinds = dict(kinds or {})
        obj.band_agree = band_agree
        obj.tag = tag
        return obj


def record(count: BandCount) -> None:
    RECORDS.append(count)


def table() -> list:
    lines = ["%-44s %8s %6s %6s %6s %6s %6s %10s" % ("comparison", "checked", "band", "accept",
                                                       "cdf", "select", "resid", "band_agree")]
    tot = [0, 0, 0, 0, 0, 0, 0]
    for r in RECORDS:
        row = [r.checked, int(r)] + [r.kinds.get(k, 0) for k in KINDS.values()] + [r.band_agree]
        tot = [a + b for a, b in zip(tot, row)]
        lines.append("%-44s %8d %6d %6d %6d %6d %6d %10d" % ((r.tag[:44],) + tuple(row)))
    lines.append("%-44s %8d %6d %6d %6d %6d %6d %10d" % (("total",) + tuple(tot)))
    return lines
