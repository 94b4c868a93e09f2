"""pytest plugin used by test_pins_catch_mutants.py (never by the library).

Before any test module is imported, it replaces the oracle's module by a
copy of its source with one planted mistake, given in the environment as
ORACLE_MUTANT = JSON [old, new] (a text that must occur exactly once in
oracle/attention.py, and its replacement). Without ORACLE_MUTANT it does
nothing, which is the control run.
"""
import json
import os
import sys
import types

import oracle
import oracle.attention as _real

_spec = os.environ.get("ORACLE_MUTANT")
if _spec:
    _old, _new = json.loads(_spec)
    with open(_real.__file__, encoding="utf-8") as _f:
        _src = _f.read()
    if _src.count(_old) != 1:
        raise RuntimeError(f"mutation site found {_src.count(_old)} times: {_old!r}")
    _mod = types.ModuleType("oracle.attention")
    _mod.__file__ = _real.__file__
    exec(compile(_src.replace(_old, _new), _real.__file__, "exec"), _mod.__dict__)
    sys.modules["oracle.attention"] = _mod
    oracle.attention = _mod
    for _name in list(vars(oracle)):
        if not _name.startswith("_") and hasattr(_mod, _name) and _name != "attention":
            setattr(oracle, _name, getattr(_mod, _name))
