"""Loading of the page-printed fixtures under tests/golden."""
import json
import math
import pathlib
import re

GOLDEN = pathlib.Path(__file__).parent / "golden"


def load(name):
    return json.loads((GOLDEN / name).read_text())


_TOKEN = re.compile(r"^(-?)(ln|sqrt)\((\d+(?:\.\d+)?)\)$")


def ev(x):
    """Evaluate a fixture entry: a number, 'ln(a)', 'sqrt(a)', '1/sqrt(a)',
    optionally with a leading minus sign."""
    if isinstance(x, (int, float)):
        return float(x)
    x = x.strip()
    if x.startswith("1/"):
        return 1.0 / ev(x[2:])
    m = _TOKEN.match(x)
    if m:
        sign = -1.0 if m.group(1) else 1.0
        fn = math.log if m.group(2) == "ln" else math.sqrt
        return sign * fn(float(m.group(3)))
    return float(x)


def ev_all(xs):
    if isinstance(xs, list):
        return [ev_all(x) for x in xs]
    return ev(xs)
