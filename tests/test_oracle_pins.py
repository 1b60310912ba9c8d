"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_every_oracle_function_declares_its_arguments():
    """ctypes passes undeclared arguments as C int: a pointer would be cut to 32 bits."""
    import re
    import subprocess
    import oracle
    lib = oracle.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", oracle._LIB], capture_output=True, text=True).stdout
    names = sorted(set(re.findall(r" T (oracle_\w+)", out)))
    assert len(names) > 40
    for name in names:
        assert getattr(lib, name).argtypes is not None, name
