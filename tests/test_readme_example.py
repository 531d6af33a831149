"""The README's usage example calls the binding as it is: every `api.*` and
block-manager call in it binds to the function's signature (its positional
arguments are exactly the required parameters, its keywords name options),
and every `api.*` name it reads exists.  CPU only: the
example is parsed, not run (running it needs a GPU)."""

import ast
import inspect
import os
import re

from paged_kv_cache_124_gb300 import api

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def _example():
    blocks = re.findall(r"```python\n(.*?)```", open(README).read(), re.S)
    assert len(blocks) == 1
    return ast.parse(blocks[0])


def _target(call):
    """The function an `api.f(...)` or `alloc.f(...)` call reaches, with the
    number of leading arguments bound implicitly (self)."""
    f = call.func
    if isinstance(f, ast.Attribute) and isinstance(f.value, ast.Name):
        if f.value.id == "api":
            return getattr(api, f.attr), 0
        if f.value.id == "alloc":
            return getattr(api.BlockAllocator, f.attr), 1
    return None, 0


def test_every_binding_call_in_the_example_binds():
    calls = [n for n in ast.walk(_example()) if isinstance(n, ast.Call)]
    checked = set()
    for c in calls:
        fn, implicit = _target(c)
        if fn is None:
            continue
        assert not any(isinstance(a, ast.Starred) for a in c.args)
        args = [object()] * (implicit + len(c.args))
        kwargs = {k.arg: object() for k in c.keywords}
        sig = inspect.signature(fn)
        sig.bind(*args, **kwargs)                        # raises TypeError on a mismatch
        # positional arguments fill exactly the required parameters (options go by keyword)
        required = [p for p in sig.parameters.values() if p.default is inspect.Parameter.empty]
        assert len(args) == len(required), "%s: %d positional arguments for %d required parameters" % (
            fn.__name__, len(args), len(required))
        checked.add(fn.__name__)
    assert {"pa_reshape_and_cache", "pa_prefill", "pa_copy_blocks", "pa_decode_append", "decode_workspace",
            "allocate", "fork", "append_slots", "build_tables", "slot_mapping", "free"} <= checked


def test_every_api_name_in_the_example_exists():
    for n in ast.walk(_example()):
        if isinstance(n, ast.Attribute) and isinstance(n.value, ast.Name) and n.value.id == "api":
            assert hasattr(api, n.attr), n.attr
