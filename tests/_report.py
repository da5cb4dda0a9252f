"""Per-session record of oracle-parity counts, printed in pytest's terminal
summary (so that the counts reach the log even under -q)."""
from __future__ import annotations

PARITY: list[tuple[str, dict]] = []


def record(name: str, summary: dict) -> None:
    PARITY.append((name, dict(summary)))
