"""Parity records of the GPU tests: per case, the requests checked, how many
the oracle flagged as near-ties and how many of those the CUDA path resolved
the other way.  ``tests/conftest.py`` prints them at the end of the run."""
RECORDS: list[dict] = []


def record(**kw) -> None:
    RECORDS.append(kw)
