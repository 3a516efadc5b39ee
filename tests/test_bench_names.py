"""bench.py runs on the GPU machine only in full, so a name that one of its
workload paths uses but never defines would surface there first.  This CPU
test resolves, with the compiler's own symbol tables, every global name any
function of bench.py reads: each must be defined at module level or be a
builtin."""
import builtins
import os
import symtable

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _walk(table):
    yield table
    for child in table.get_children():
        yield from _walk(child)


def test_bench_functions_use_only_defined_globals():
    path = os.path.join(ROOT, "bench.py")
    top = symtable.symtable(open(path).read(), path, "exec")
    defined = {s.get_name() for s in top.get_symbols() if s.is_assigned() or s.is_imported()}
    defined |= set(dir(builtins))
    missing = []
    for t in _walk(top):
        if t.get_type() != "function":
            continue
        for s in t.get_symbols():
            if s.is_global() and s.is_referenced() and s.get_name() not in defined:
                missing.append(f"{t.get_name()}: {s.get_name()}")
    assert not missing, missing
