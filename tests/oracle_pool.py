"""Worker side of gpu_util.oracle_map: runs one oracle function on one chunk.
Imports only numpy and the oracle, so spawned workers start quickly."""
import oracle


def call(args):
    name, arrays, kwargs = args
    return getattr(oracle, name)(*arrays, **kwargs)
