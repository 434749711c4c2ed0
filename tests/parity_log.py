"""Parity figures printed by the GPU tests, collected so that the end of a pytest
run repeats them in one place (pytest hides a passing test's output)."""
import os

LINES = []


def record_parity(line: str) -> None:
    print(line)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0].split("::")[-1]
    LINES.append(f"{test}: {line}" if test else line)
