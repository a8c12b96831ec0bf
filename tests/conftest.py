import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


# Modules run after all others, in this order (the rest keep pytest's order).
RUN_LAST = ("test_no_alloc.py",)


def pytest_collection_modifyitems(session, config, items):
    def rank(item):
        name = os.path.basename(str(item.fspath))
        return RUN_LAST.index(name) + 1 if name in RUN_LAST else 0

    items.sort(key=rank)  # stable: the order within each rank is kept
